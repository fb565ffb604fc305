// The standalone tcgen05 state pass (the chain body is in chain_umma.cuh): one CTA per (session, v-head, slice
// of d_v) chain, launched after the call's prologue kernel.
#include "chain_umma.cuh"

namespace gdn {

template <int N>
__global__ void __launch_bounds__(kChainWorkThreads, 1) chain_umma_kernel(const __grid_constant__ LaunchCommon p, int64_t ch) {
    extern __shared__ __align__(1024) unsigned char sm[];
    grid_dep_launch();   // the next call's prologue may take SMs as this kernel's CTAs leave
    grid_dep_wait();     // the records of this call, the state and the conv state
    RecordsWritten ready;
    chain_run<N, kChainWorkThreads, 8>(p, ch, sm, blockIdx.x, ready);
}

template <int N>
static cudaError_t launch_cols(const LaunchCommon &p, int64_t ch, cudaStream_t st) {
    constexpr size_t smem = UChainPlan<N>::kBytes;
    auto k = chain_umma_kernel<N>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = gdn_launch_pdl(k, p.n_sess * p.Hv * (128 / N), kChainWorkThreads, smem, st, p, ch);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace gdn

// 32 columns per CTA (4 CTAs per chain) while the launch fits one wave: the shortest dependent step for a few
// chains; 64 or 128 once it would not, where the per-chain operand traffic and throughput count.
int gdn_chain_umma_cols(int n_chains_of_128, int sms) {
    if (4 * n_chains_of_128 <= sms) return 32;
    if (2 * n_chains_of_128 <= sms) return 64;
    return 128;
}

cudaError_t gdn_launch_chain_umma(const gdn::LaunchCommon &p, int64_t ch, cudaStream_t st, int cols) {
    if (cols == 0) {
        int sms = 1;
        cudaError_t e = gdn_sm_count(&sms);
        if (e != cudaSuccess) return e;
        cols = gdn_chain_umma_cols(p.n_sess * p.Hv, sms);
    }
    switch (cols) {
        case 32: return gdn::launch_cols<32>(p, ch, st);
        case 64: return gdn::launch_cols<64>(p, ch, st);
        default: return gdn::launch_cols<128>(p, ch, st);
    }
}
