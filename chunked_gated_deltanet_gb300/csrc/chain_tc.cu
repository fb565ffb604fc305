// Sequential state pass and outputs on tensor cores (bf16-input path): one CTA
// per (session, v-head, slice of d_v) chain (the pieces are in chain_tc.cuh),
// 8 warps. Block b+1's operands load while block b computes. Every wait on an
// mbarrier is bounded: on timeout the CTA records it in the device error word,
// waits (bounded) for its copies in flight, and returns. The CTA also commits
// its share of the session's conv state.
#include "chain_tc.cuh"

__device__ unsigned int g_gdn_device_error;

namespace gdn {

template <int D, int DS>
__global__ void __launch_bounds__(kThreads, 1) chain_tc_kernel(const __grid_constant__ LaunchCommon p, int64_t ch) {
    extern __shared__ __align__(16) float smem[];
    Chain<D, DS> c(p, smem, blockIdx.x);
    const int t = threadIdx.x, nb = c.nb;
    grid_dep_launch();   // the next call's prologue may take SMs as this kernel's CTAs leave
    if (t == 0) c.init_bars();
    grid_dep_wait();     // the records of this call, the state and the conv state
    if (t == 0) {   // the first block's copies go out first; the conv commit and the state load overlap them
        if (nb > 0) {
            c.issue(0);
            if constexpr (Chain<D, DS>::kSplit) c.issue_wq(0);
        }
    }
    c.conv_commit(ch);
    c.load_state();
    __syncthreads();
    int timed_out = 0;
    for (int b = 0; b < nb; ++b) {
        if (t == 0 && b + 1 < nb) c.issue(b + 1);   // the other stage was released at the end of step b-1
        const bool to = c.step(b);
        // (C) state copy updated; this stage is free for block b+2; uniform timeout decision
        if (__syncthreads_or(to)) {   // every thread leaves at the same step
            timed_out = b + 1;
            break;
        }
    }
    if (timed_out) {   // record the timeout, then wait (bounded) for this CTA's copies still in flight
        if (t == 0) {
            atomicOr(p.err, 1u);
            c.drain(timed_out - 1, timed_out < nb);
        }
        __syncthreads();
        return;
    }
    c.finish();
}

template <int D, int DS>
static cudaError_t launch(const LaunchCommon &p, int64_t ch, cudaStream_t st) {
    constexpr size_t smem = ChainPlan<D, DS>::bytes();
    static_assert(smem <= 227 * 1024, "shared memory");
    auto k = chain_tc_kernel<D, DS>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = gdn_launch_pdl(k, p.n_sess * p.Hv * (D / DS), kThreads, smem, st, p, ch);
    return e != cudaSuccess ? e : cudaGetLastError();
}

template <int D>
static cudaError_t launch_d(const LaunchCommon &p, int64_t ch, cudaStream_t st) {
    // 16 columns per CTA while the launch fits one wave (one CTA per SM): the shortest step for a few
    // chains; 32 columns once it would not, where throughput counts. The arithmetic of every state
    // element is the same in both (same MMAs, same accumulation order), so results do not depend on it.
    int sms = 1;
    if (gdn_sm_count(&sms) != cudaSuccess) sms = 1;
    if ((int64_t)p.n_sess * p.Hv * (D / kSliceCols) > sms) return launch<D, 2 * kSliceCols>(p, ch, st);
    return launch<D, kSliceCols>(p, ch, st);
}

}  // namespace gdn

cudaError_t gdn_launch_chain_tc(const gdn::LaunchCommon &p, int D, int64_t ch, cudaStream_t st) {
    return D == 64 ? gdn::launch_d<64>(p, ch, st) : gdn::launch_d<128>(p, ch, st);
}

#include <mutex>

cudaError_t gdn_device_error_word(unsigned int **out) {
    static std::mutex mu;
    static unsigned int *addr[64] = {};
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *a = nullptr;
        e = cudaGetSymbolAddress(&a, g_gdn_device_error);
        if (e != cudaSuccess) return e;
        addr[dev] = static_cast<unsigned int *>(a);
    }
    *out = addr[dev];
    return cudaSuccess;
}

cudaError_t gdn_sm_count(int *out) {
    static std::mutex mu;
    static int count[64] = {};
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!count[dev]) {
        e = cudaDeviceGetAttribute(&count[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
    }
    *out = count[dev];
    return cudaSuccess;
}

cudaError_t gdn_take_device_error(unsigned int *out, cudaStream_t st) {
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(out, g_gdn_device_error, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_gdn_device_error, &zero, sizeof(unsigned int));
}
