// The standalone tcgen05 prologue kernel (the task body is in prologue_umma.cuh): persistent, one CTA per
// SM over the launch's (block, q/k head) tasks.
#include "prologue_umma.cuh"

namespace gdn {

// kAct: SiLU after the causal conv (LaunchCommon::act), as a template parameter so that the instantiation
// without it keeps its loop compact.
template <bool kAct>
__global__ void __launch_bounds__(kUmmaPrepThreads, 1)
    prep_umma_kernel(const __grid_constant__ LaunchCommon p, int64_t ch) {
    extern __shared__ __align__(1024) unsigned char sm[];
    UmmaCtl *ctl = reinterpret_cast<UmmaCtl *>(sm + up::OFF_BAR);
    if (threadIdx.x == 32 && (int)blockIdx.x < p.nblk * p.Hk) {
        // The first task's input tiles and gates into L2 while this CTA waits for earlier work. A prefetch only
        // places lines in L2, the point of coherence, so a write that lands later still wins.
        const int blk = (int)blockIdx.x % p.nblk, hk = (int)blockIdx.x / p.nblk;
        const SessRef s = p.s[find_session(p, blk)];
        const int pos0 = (blk - s.blk0) * kBlock, row0 = (int)(s.row0 + pos0);
        tma_prefetch_2d(&p.tm_q, hk * up::D, row0);
        tma_prefetch_2d(&p.tm_k, hk * up::D, row0);
        for (int gi = 0; gi < p.G; ++gi) tma_prefetch_2d(&p.tm_v, (hk * p.G + gi) * up::D, row0);
        prefetch_gates(p, row0, min(kBlock, s.n - pos0));
    }
    if ((threadIdx.x >> 5) == 0) {
        tmem_alloc(&ctl->tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tslot;
    grid_dep_launch();   // the state kernel may take SMs as this kernel's CTAs leave
    grid_dep_wait();     // inputs and conv state of this call, written by earlier work
    StridedTasks src{(int)blockIdx.x, p.nblk * p.Hk};
    prologue_run<kAct>(p, ch, sm, ctl, tmem, src);
    tc_fence_after();
    if ((threadIdx.x >> 5) == 0) tmem_dealloc(tmem, 512);
}

}  // namespace gdn

cudaError_t gdn_launch_prep_umma(const gdn::LaunchCommon &p, int64_t ch, cudaStream_t st) {
    using namespace gdn;
    auto k = p.act ? prep_umma_kernel<true> : prep_umma_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)up::SMEM);
    if (e != cudaSuccess) return e;
    int sms = 1;   // one persistent CTA per SM (shared memory allows no more), over nblk x Hk tasks
    if ((e = gdn_sm_count(&sms)) != cudaSuccess) return e;
    const int ntask = p.nblk * p.Hk;
    e = gdn_launch_pdl(k, ntask < sms ? ntask : sms, kUmmaPrepThreads, up::SMEM, st, p, ch);
    return e != cudaSuccess ? e : cudaGetLastError();
}
