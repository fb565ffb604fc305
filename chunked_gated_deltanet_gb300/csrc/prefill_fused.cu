// The one-launch prefill (bf16 inputs, d = 128) for calls with few chains: one persistent CTA per SM.
//
// CTAs [0, n_chain) run the state pass, one chain each (session, v-head, 64 columns of d_v; chain_umma.cuh), on
// 8 worker warps; warp 8 polls the records' publication and issues the copies, warps 9-15 commit the conv state.
// (All 16 warps as workers, with the polls inside the step, measured slower.)
// The other CTAs run the prologue (prologue_umma.cuh) over the call's (64-token block, q/k head) tasks in
// block order, CTA j taking tasks j, j + P, j + 2P, ... of the P prologue CTAs. A task's record, once
// written, is published by a release store of this call's epoch into its flag; the chain CTA that needs it
// polls the flag with acquire loads (bounded, with a short sleep between polls), orders that view with its
// bulk-copy proxy and then copies the record in. So the state pass of a block starts as soon as its records
// exist, and the prologue's tasks run beside the state passes instead of before them. Every CTA of the launch
// is resident at once (one CTA per SM, grid = SM count), and the chains wait only on prologue CTAs of the same
// launch, which never wait on them.
//
// Each record and each state element is computed by the same code, in the same order, as in the two-launch
// path (prologue kernel, then state kernel), so both paths give the same bits. The conv state is committed
// by the chain CTAs once the session's first block is published (its halo reads of the old conv state are
// then done).
#include "chain_umma.cuh"
#include "prologue_umma.cuh"

namespace gdn {

struct FusedArgs {
    unsigned long long *flags;   // [nblk][Hk], publication words
    unsigned long long epoch;    // this call's value of a published flag
    int n_chain;                 // chain CTAs (the first ones of the grid)
};

// Prologue task source of the one-launch prefill: static striding over the prologue CTAs, block-major task
// numbering (LaunchCommon::task_block_major), and a publication of each completed task.
struct FusedTasks {
    int tau, stride, ntask;
    unsigned long long *flags;
    unsigned long long epoch;
    int Hk;
    __device__ __forceinline__ int first() { return tau < ntask ? tau : -1; }
    __device__ __forceinline__ int next() { tau += stride; return tau < ntask ? tau : -1; }
    __device__ __forceinline__ int peek() const { return tau + stride < ntask ? tau + stride : -1; }
    // called by every thread after the CTA barrier that follows the task's last record store
    __device__ __forceinline__ void done(int blk, int hk) {
        if (threadIdx.x == 0) {
            fence_proxy_async_global();
            __threadfence();
            st_release_gpu(flags + (int64_t)blk * Hk + hk, epoch);
        }
    }
};

// A chain's wait for a block's record: polls its flag with acquire loads, at most `limit` times.
struct FlagReady {
    const unsigned long long *flags;
    unsigned long long epoch;
    int Hk;
    long long limit;
    __device__ __forceinline__ bool operator()(int blk, int hk) const {
        const unsigned long long *f = flags + (int64_t)blk * Hk + hk;
        for (long long i = 0; i < limit; ++i) {
            if (ld_acquire_gpu(f) == epoch) {
                fence_proxy_async_global();   // the bulk copies that follow read what the flag published
                return true;
            }
            __nanosleep(32);
        }
        return false;
    }
};

template <bool kAct>
__global__ void __launch_bounds__(kUmmaPrepThreads, 1)
    prefill_fused_kernel(const __grid_constant__ LaunchCommon p, int64_t ch, const FusedArgs f) {
    extern __shared__ __align__(1024) unsigned char sm[];
    grid_dep_launch();   // every CTA of this launch has started: the next kernel may take SMs as ours leave
    if ((int)blockIdx.x >= f.n_chain && threadIdx.x == 32) {   // a prologue CTA's first task's inputs into L2
        const int pc = (int)blockIdx.x - f.n_chain;
        if (pc < (p.nblk - p.blk_lo) * p.Hk) prefetch_task_inputs(p, p.blk_lo + pc / p.Hk, pc % p.Hk);
    }
    grid_dep_wait();     // the states, conv states and workspace of earlier work
    if ((int)blockIdx.x < f.n_chain) {
        FlagReady ready{f.flags, f.epoch, p.Hk, p.wait_limit};
        chain_run<kFusedCols, kUmmaPrepThreads, 8>(p, ch, sm, blockIdx.x, ready);
        return;
    }
    UmmaCtl *ctl = reinterpret_cast<UmmaCtl *>(sm + up::OFF_BAR);
    if ((threadIdx.x >> 5) == 0) {
        tmem_alloc(&ctl->tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tslot;
    const int pc = (int)blockIdx.x - f.n_chain, np = (int)gridDim.x - f.n_chain;
    FusedTasks src{pc, np, (p.nblk - p.blk_lo) * p.Hk, f.flags, f.epoch, p.Hk};
    prologue_run<kAct>(p, ch, sm, ctl, tmem, src);
    tc_fence_after();
    if ((threadIdx.x >> 5) == 0) tmem_dealloc(tmem, 512);
}

}  // namespace gdn

cudaError_t gdn_launch_prefill_fused(const gdn::LaunchCommon &p, int64_t ch, unsigned long long *flags,
                                     unsigned long long epoch, int n_chain, cudaStream_t st) {
    using namespace gdn;
    constexpr size_t chain_smem = UChainPlan<kFusedCols, 8>::kBytes;
    constexpr size_t smem = up::SMEM > chain_smem ? up::SMEM : chain_smem;
    static_assert(smem <= 227 * 1024, "shared memory");
    auto k = p.act ? prefill_fused_kernel<true> : prefill_fused_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int sms = 1;
    if ((e = gdn_sm_count(&sms)) != cudaSuccess) return e;
    if (n_chain < 1 || n_chain >= sms) return cudaErrorInvalidValue;
    const FusedArgs f{flags, epoch, n_chain};
    e = gdn_launch_pdl(k, sms, kUmmaPrepThreads, smem, st, p, ch, f);
    return e != cudaSuccess ? e : cudaGetLastError();
}
