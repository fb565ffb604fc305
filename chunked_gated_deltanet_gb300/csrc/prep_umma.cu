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
    const int nbt = p.nblk - p.blk_lo;   // blocks of this launch's tasks
    if (threadIdx.x == 32 && (int)blockIdx.x < nbt * p.Hk)   // the first task's inputs, while waiting below
        prefetch_task_inputs(p, p.blk_lo + (int)blockIdx.x % nbt, (int)blockIdx.x / nbt);
    if ((threadIdx.x >> 5) == 0) {
        tmem_alloc(&ctl->tslot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctl->tslot;
    // A launch over all of a call's blocks waits for earlier work (inputs, conv state, and the state pass
    // of the call before, which reads the workspace) and only then lets the next kernel launch, so that
    // everything launched after it starts after that work too. A launch over the last blocks only
    // (blk_lo > 0) follows the state pass of the call's first blocks and runs beside it: it needs neither
    // the conv state (none of its blocks is a session's first) nor anything that state pass writes, and
    // writes other records than it reads, so it waits for it only at its end; the second state pass, which
    // waits for this launch, thereby starts after the first.
    const bool tail = p.blk_lo > 0;
    if (!tail) grid_dep_wait();
    grid_dep_launch();   // the next kernel may take SMs as this kernel's CTAs leave
    StridedTasks src{(int)blockIdx.x, nbt * p.Hk};
    prologue_run<kAct>(p, ch, sm, ctl, tmem, src);
    if (tail) grid_dep_wait();
    tc_fence_after();
    if ((threadIdx.x >> 5) == 0) tmem_dealloc(tmem, 512);
}

}  // namespace gdn

cudaError_t gdn_launch_prep_umma(const gdn::LaunchCommon &p, int64_t ch, cudaStream_t st, int max_ctas) {
    using namespace gdn;
    auto k = p.act ? prep_umma_kernel<true> : prep_umma_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)up::SMEM);
    if (e != cudaSuccess) return e;
    int sms = 1;   // one persistent CTA per SM (shared memory allows no more), over nblk x Hk tasks
    if ((e = gdn_sm_count(&sms)) != cudaSuccess) return e;
    if (max_ctas > 0 && max_ctas < sms) sms = max_ctas;
    const int ntask = (p.nblk - p.blk_lo) * p.Hk;
    e = gdn_launch_pdl(k, ntask < sms ? ntask : sms, kUmmaPrepThreads, up::SMEM, st, p, ch);
    return e != cudaSuccess ? e : cudaGetLastError();
}
