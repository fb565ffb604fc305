// Internal definitions shared by the library's kernels and its C ABI layer.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

constexpr int kBlock = 64;           // tokens per compute block (divides every grid C)
constexpr int kLaunchSessions = 64;  // sessions described by one launch's parameters
constexpr int kThreads = 256;

// One session's slice of a launch.
struct SessRef {
    int64_t row0;    // first row of the session's tokens in the packed inputs / outputs
    int32_t n;       // tokens processed for this session in this call
    int32_t blk0;    // index of its first 64-token block in the launch's block numbering
    float *S;        // fp32 [Hv][D][D] state (transposed): the result goes here
    void *conv;      // in_dtype [3][ch] conv state: the result goes here
    const float *S0;      // the state the call starts from (S itself, or a shared prefix's state)
    const void *conv0;    // the conv state it starts from (conv itself, or the prefix's)
    float *S_cap;         // optional checkpoint: the final state is also written here (null: none)
    void *conv_cap;       // and the final conv state here
};

struct LaunchCommon {
    const void *xq, *xk, *xv;   // packed inputs
    const float *g, *beta;      // [rows][Hv]
    const void *conv_w;         // [ch][4]
    void *out;                  // [rows][Hv][D]
    float *ws_qk;               // fp32 path: [nblk][Hk][2][64][D] q_hat, k_hat
    float *ws_wu;               // per (block, v-head) record: fp32 path [wu_floats] W, U, P, gamma; bf16 paths
                                // the layouts of their state kernels (rec16::kBytes for d = 128)
    int Hk, Hv, G;
    int act, out_bf16;
    float q_scale, eps;
    int n_sess;
    int nblk;                   // total blocks of this launch
    int blk_lo;                 // tcgen05 prologue: > 0 runs the tasks of blocks [blk_lo, nblk) only, beside the
                                // state pass launched before it, and waits for that one at its end (see prep_umma.cu)
    int task_block_major;       // tcgen05 prologue: tasks numbered block first (the one-launch prefill), else head first
    long long wait_limit;       // polls before a bounded mbarrier wait gives up
    unsigned int *err;          // device error word (bit 0: a bounded wait ran out)
    int debug_skip_first_copy;  // test hook: 1 = the state kernel, 2 = the tcgen05 prologue never issues its first copy
    SessRef s[kLaunchSessions];
    // the state kernel's session order: chain CTAs are numbered session order[0] first (the caller lists
    // the longest first, so that the longest chains start first and the launch packs well)
    unsigned char order[kLaunchSessions];
    // 2-D tensor maps over xq [rows][Hk D], xk [rows][Hk D], xv [rows][Hv D] (bf16, boxes of 64 rows x 128
    // channels) for the tcgen05 prologue's input copies; encoded by the host per call, unused elsewhere
    CUtensorMap tm_q, tm_k, tm_v;
};

// Per-(block, v-head) record in the workspace: W [64][D], U [64][D], P [64][64], gamma [64].
__host__ __device__ constexpr int64_t wu_floats(int D) { return 2LL * kBlock * D + kBlock * kBlock + kBlock; }
__host__ __device__ constexpr int64_t qk_floats(int D) { return 2LL * kBlock * D; }
// Tensor-core path, per-(block, v-head) record (floats), laid out in the order
// the state kernel's m16n8k8 fragments read it (g = lane / 4, t = lane % 4):
//   [0, 128 D)      A fragments of [W; Qe] (128 x D): [m-tile 0..7][k-step 0..D/8-1][lane][4]
//   [128 D, 192 D)  A fragments of K_tilde^T (D x 64): [m-tile 0..D/16-1][k-step 0..7][lane][4]
//   [192 D, 256 D)  C fragments of U (64 x D) by 16-column slice: [slice][m-tile 0..3][n-tile 0..1][lane][4]
//   [256 D, 320 D)  C fragments of O_intra, same order
//   [320 D]         e^{gamma_63}, then padding to 320 D + 16
// [W; Qe] and K_tilde are stored rounded to tf32; U and O_intra are fp32.
__host__ __device__ constexpr int64_t rec_floats(int D) { return 320LL * D + 16; }
constexpr int kSliceCols = 16;  // d_v columns per state-kernel CTA

// Index of element (r, k) of an A operand with K columns inside its fragment-ordered array.
__device__ __forceinline__ int afrag_index(int r, int k, int K) {
    const int rr = r & 15, kk = k & 7;
    const int lane = 4 * (rr & 7) + (kk & 3), f = (rr >> 3) + 2 * (kk >> 2);
    return (((r >> 4) * (K >> 3) + (k >> 3)) * 32 + lane) * 4 + f;
}
// Index of element (i, c) of a 64 x D accumulator stored by 16-column slices of C fragments.
__device__ __forceinline__ int cfrag_slice_index(int i, int c) {
    const int sl = c >> 4, cc = c & 15, ri = i & 15;
    const int lane = 4 * (ri & 7) + ((cc & 7) >> 1), f = 2 * (ri >> 3) + (cc & 1);
    return ((((sl * 4 + (i >> 4)) * 2 + (cc >> 3)) * 32 + lane) * 4 + f);
}

// fp16 record of the tcgen05 path (bf16 inputs, d_k = d_v = 128), one per (64-token block, v-head), written
// by the prologue in the layouts the tcgen05 state pass reads straight from shared memory. Offsets in bytes.
// A core matrix is 8 rows x 16 bytes (8 fp16), stored as 128 contiguous bytes.
namespace rec16 {
constexpr uint32_t kWQ = 0;         // [W; Qe], 128 x 128: A operand of [W; Qe] S^T, K-major cores, LBO 128 (along K),
                                    // SBO 2048 (along M)
constexpr uint32_t kKT = 32768;     // K_tilde^T, 128 (d_k) x 64 (tokens): A operand of K_tilde^T U', MN-major cores
                                    // (a core row is 8 d_k channels of one token), LBO 2048 (along K), SBO 128 (along M)
constexpr uint32_t kU = 49152;      // U, 64 x 128, as [column / 8][row][column % 8]: 1 KB per 8 columns
constexpr uint32_t kO = 65536;      // O_intra, the same layout
constexpr uint32_t kEg = 81920;     // e^{gamma_63} (fp32)
constexpr uint32_t kBytes = 82048;  // the record's stride (a multiple of 128 bytes)
__host__ __device__ constexpr uint32_t wq(int r, int k) {
    return (uint32_t)(r >> 3) * 2048u + (uint32_t)(k >> 3) * 128u + (uint32_t)(r & 7) * 16u + (uint32_t)(k & 7) * 2u;
}
__host__ __device__ constexpr uint32_t kt(int d, int j) {
    return kKT + (uint32_t)(d >> 3) * 128u + (uint32_t)(j >> 3) * 2048u + (uint32_t)(j & 7) * 16u + (uint32_t)(d & 7) * 2u;
}
__host__ __device__ constexpr uint32_t uo(int i, int c) { return (uint32_t)(c >> 3) * 1024u + (uint32_t)i * 16u + (uint32_t)(c & 7) * 2u; }
}  // namespace rec16

template <typename T> __device__ __forceinline__ float to_f(T x);
template <> __device__ __forceinline__ float to_f<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ int find_session(const LaunchCommon &p, int blk) {
    int s = 0;
    while (s + 1 < p.n_sess && p.s[s + 1].blk0 <= blk) ++s;
    return s;
}

// Release / acquire of a 64-bit flag at GPU scope (the one-launch prefill's per-record flags).
__device__ __forceinline__ void st_release_gpu(unsigned long long *a, unsigned long long v) {
    asm volatile("st.release.gpu.global.u64 [%0], %1;\n" ::"l"(a), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_acquire_gpu(const unsigned long long *a) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];\n" : "=l"(v) : "l"(a) : "memory");
    return v;
}
// Orders this thread's generic-proxy view of global memory with its async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;\n" ::: "memory"); }

// Programmatic dependent launch: a kernel launched with programmatic stream serialization may start while
// the kernel before it in the stream is still running. grid_dep_launch() lets the next kernel start (its
// CTAs take SMs as ours leave); grid_dep_wait() returns once every earlier kernel has completed and its
// memory operations are visible, so it must precede any read of data earlier work wrote (and any write
// earlier work may still read). Both are no-ops without a programmatic predecessor or successor.
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); }
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

// Causal conv of one channel over a 64-row block, fixed fma order (oldest tap first).
// x_at(i) returns the raw input at block row i (i in [-3, n)), zero is used past n.
template <typename InT>
__device__ __forceinline__ float conv_tap(const float w[4], float xm3, float xm2, float xm1, float x0, int act) {
    float acc = w[0] * xm3;
    acc = fmaf(w[1], xm2, acc);
    acc = fmaf(w[2], xm1, acc);
    acc = fmaf(w[3], x0, acc);
    if (act) acc = acc / (1.0f + expf(-acc));
    return acc;
}

}  // namespace gdn

// Reads and clears the device error word after synchronising the stream (bit 0: a bounded wait ran out).
cudaError_t gdn_take_device_error(unsigned int *out, cudaStream_t st);
// Device address of the error word on the current device (looked up once per device).
cudaError_t gdn_device_error_word(unsigned int **out);

// Number of SMs of the current device (looked up once per device).
cudaError_t gdn_sm_count(int *out);

// Launches kernel<<<grid, block, smem, st>>>(args...) with programmatic stream serialization (the kernel
// calls grid_dep_wait before touching data of earlier work).
template <class... K, class... A>
cudaError_t gdn_launch_pdl(void (*kernel)(K...), dim3 grid, unsigned block, size_t smem, cudaStream_t st,
                           A &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<A &&>(args)...);
}

// Sets the message gdn_last_error() returns on this host thread (library-internal).
void gdn_internal_set_error(const char *msg);

// Launchers (host). Each returns cudaGetLastError() after its launch.
cudaError_t gdn_launch_prep(const gdn::LaunchCommon &p, int D, int in_bf16, int64_t ch, cudaStream_t st);
cudaError_t gdn_launch_state(const gdn::LaunchCommon &p, int D, cudaStream_t st);
cudaError_t gdn_launch_prep_tc(const gdn::LaunchCommon &p, int D, int64_t ch, cudaStream_t st);
// max_ctas: at most that many CTAs (0: one per SM)
cudaError_t gdn_launch_prep_umma(const gdn::LaunchCommon &p, int64_t ch, cudaStream_t st, int max_ctas = 0);
cudaError_t gdn_launch_chain_tc(const gdn::LaunchCommon &p, int D, int64_t ch, cudaStream_t st);
// The one-launch prefill (bf16, d = 128): n_chain chain CTAs (64 d_v columns each) beside prologue CTAs on every
// other SM; flags: [nblk][Hk] publication words in the workspace, epoch: this call's value for them.
cudaError_t gdn_launch_prefill_fused(const gdn::LaunchCommon &p, int64_t ch, unsigned long long *flags,
                                     unsigned long long epoch, int n_chain, cudaStream_t st);
constexpr int kFusedCols = 64;   // d_v columns per chain CTA of the one-launch prefill
// The tcgen05 state pass over fp16 records (d = 128); cols: d_v columns per CTA (32, 64 or 128; 0 chooses by the
// launch's chain count, gdn_chain_umma_cols)
cudaError_t gdn_launch_chain_umma(const gdn::LaunchCommon &p, int64_t ch, cudaStream_t st, int cols = 0);
int gdn_chain_umma_cols(int n_chains_of_128, int sms);
cudaError_t gdn_launch_conv_commit(const gdn::LaunchCommon &p, int D, int in_bf16, int64_t ch, cudaStream_t st);
cudaError_t gdn_launch_copy(void *dst0, const void *src0, size_t bytes0, void *dst1, const void *src1,
                            size_t bytes1, cudaStream_t st);
// chunk: the index of this launch among the launches of one decode call (64 sessions each)
cudaError_t gdn_launch_decode(const gdn::LaunchCommon &p, int D, int in_bf16, int64_t ch, int chunk, cudaStream_t st);
cudaError_t gdn_launch_gates(const float *a, const float *b, const float *A_log, const float *dt_bias, int64_t n,
                             int Hv, float *g, float *beta, cudaStream_t st);
