// Prologue + WY/UT transform on the 5th-generation tensor core (tcgen05,
// accumulators in TMEM), bf16 inputs, d_k = d_v = 128, as a task runner that a
// kernel calls: a task is one (64-token block, q/k head), for each of the
// head's G v-heads.
//
// The quantities are those of the mma.sync prologue (prep_tc.cu):
//   conv (kernel 4, halo from the conv state at a call's first block), L2 norm
//   gamma = cumulative log-decay in the block
//   A_ij = beta_i e^{gamma_i - gamma_j} (K K^T)_ij (j < i),  T = (I + A)^{-1}
//   W = T diag(beta e^gamma) K_hat,  U = T diag(beta) V
//   P_ij = e^{gamma_i - gamma_j} (Q K^T)_ij (j <= i)
//   Qe = diag(e^gamma) Q_hat - P W,  O_intra = P U,  K_tilde = diag(e^{gamma_63 - gamma_j}) K_hat
// and the record goes out in fp16, in the operand layouts the state pass copies
// straight into shared memory (common.cuh, rec16).
//
// The products run as tcgen05 MMAs of M = 128, issued by one thread, with fp32
// accumulation. [Q_hat; K_hat] K_hat^T takes bf16 hi/lo operand pairs (hi*hi +
// hi*lo + lo*hi, about 16 significant bits per operand): the dot product of two
// nearly orthogonal unit vectors cancels, and one rounding of the operands
// would lose it. P T and the main product take single fp16 operands (11
// significant bits, the precision of the record the state pass reads). P W = (P T) Bk and P U = (P T) Bv, so
// stacking [T; P T] as the A operand gives all four 64 x 128 results of the
// block in one product whose every accumulator row is used:
//   [Q_hat; K_hat] K_hat^T               N = 64,  K = 128 -> TMEM columns 0..63 (kept for every v-head)
//   P T                                  N = 64,  K = 64  -> TMEM columns 64..127 (rows 64..127 unused)
//   [T; P T] [beta e^gamma K_hat | beta V] N = 256, K = 64 -> TMEM columns 256..511: [W U; P W P U]
// Operands live in shared memory in the no-swizzle layouts of umma.cuh: the
// row-ordered operands (q_hat, k_hat, P, T, P T) K-major, the token-by-channel
// B operands MN-major, so that every producer writes whole 16-byte
// core-matrix rows. The triangular inverse stays in fp32: substitution on the
// CUDA cores for its 16 x 16 diagonal blocks, tf32 mma.sync for the
// blocked products. The input tiles arrive as 2-D tensor copies (one per tile)
// plus three single-row halo copies, on an mbarrier: a task's tiles are
// copied in during the inverse of the task before it (their region is their
// own), by warps that are idle there. Every wait is bounded, and on a timeout the CTA
// records it in the device error word, waits (bounded) for what it has in
// flight and returns (the kernel then frees its TMEM).
#pragma once
#include "common.cuh"
#include "mma.cuh"
#include "umma.cuh"

namespace gdn {

constexpr int kUmmaPrepThreads = 512;

namespace up {   // shared-memory plan, bytes
constexpr int D = 128;
constexpr uint32_t AQ_LBO = 144, AQ_SBO = 16 * AQ_LBO;    // [q_hat; k_hat], K-major, K = 128, 16-byte gap between K cores
constexpr uint32_t AQ_BYTES = 16 * AQ_SBO;                  // 128 rows
constexpr uint32_t B_LBO = 128, B_SBO = 8 * B_LBO + 16;     // fp16 [beta e^gamma k_hat | beta v], MN-major, N = 256, K = 64
constexpr uint32_t B_BYTES = 32 * B_SBO;
constexpr uint32_t K64_LBO = 128, K64_SBO = 8 * K64_LBO;    // K = 64 fp16 operands: P, [T; P T] (K-major), T (MN-major)
constexpr uint32_t R64_BYTES = 8 * K64_SBO;                 // 64 rows (or 64 columns) of a K = 64 operand
constexpr int LT = kBlock + 4;                              // fp32 A and T row pitch (floats)
constexpr uint32_t OFF_AQH = 0, OFF_AQL = AQ_BYTES;
constexpr uint32_t OFF_BH = 2 * AQ_BYTES;                    // B operand
constexpr uint32_t OFF_PH = OFF_BH + B_BYTES;                // P, K-major
constexpr uint32_t OFF_TBH = OFF_PH + R64_BYTES;             // T, MN-major (B of P T)
constexpr uint32_t OFF_AF = OFF_TBH + R64_BYTES;             // fp32 A (input of the inverse)
constexpr uint32_t OFF_TF = OFF_AF + 4 * kBlock * LT;        // fp32 T
constexpr uint32_t OFF_MT = OFF_TF + 4 * kBlock * LT;        // 2 x 16 x 24 inverse scratch
constexpr uint32_t OFF_ATH = OFF_AF;                         // [T; P T], K-major, over A and T
constexpr uint32_t OFF_SMALL = OFF_MT + 4 * 2 * 16 * 24;     // gamma, beta, e^gamma
constexpr uint32_t W_BYTES = D * 4 * 2;                      // conv weights of one head's channels (bf16 [D][4])
constexpr uint32_t OFF_W = OFF_SMALL + 4 * 3 * kBlock;       // q, k, v conv weights
constexpr uint32_t RAW_ROW = 2 * D, RAW_TILE = (kBlock + 3) * RAW_ROW;
constexpr uint32_t TILE_BYTES = RAW_TILE + W_BYTES;          // one staged tile: 64 + 3 rows and its weights
constexpr uint32_t OFF_RAW = OFF_W + 3 * W_BYTES;            // raw input tiles, a region of their own: the next
                                                             // task's copies land while this one still computes
constexpr uint32_t OFF_BAR = OFF_RAW + 3 * RAW_TILE;         // the control words (UmmaCtl) of the standalone kernel
constexpr uint32_t OFF_SESS = OFF_BAR + 32;                  // the launch's sessions (SessLite), read per task
constexpr uint32_t OFF_NEXT = OFF_SESS + 24 * kLaunchSessions;   // the next task, for every thread
constexpr uint32_t SMEM = OFF_NEXT + 64;
static_assert(OFF_ATH + 2 * R64_BYTES <= OFF_MT, "[T; P T] must fit over A and T");
static_assert(OFF_RAW % 128 == 0 && RAW_TILE % 128 == 0, "tensor-copy destinations 128-byte aligned");
// the P T product reads 128 A rows from P's region: the 64 rows after it (unused results) are T's operand
static_assert(OFF_PH + 2 * R64_BYTES <= OFF_AF, "rows read past P");
static_assert(SMEM <= 227 * 1024, "shared memory");
}  // namespace up

// What a task needs of its session, copied into shared memory once per CTA.
struct SessLite {
    int64_t row0;         // first row of the session's tokens
    const void *conv0;    // the conv state it starts from
    int32_t n, blk0;      // tokens of this call, first block
};
static_assert(sizeof(SessLite) == 24, "session entry");

// Control words of the prologue, kept apart from its operand plan.
struct UmmaCtl {
    uint64_t bar[2];   // [0] input copies, [1] MMA groups
    uint32_t tslot;    // TMEM allocation result
};

// A persistent CTA's tasks: blockIdx.x, + gridDim.x, ... of the launch's (nblk - blk_lo) x Hk tasks, task
// tau = (block blk_lo + tau % (nblk - blk_lo), q/k head tau / (nblk - blk_lo)) (or, with task_block_major,
// (block blk_lo + tau / Hk, q/k head tau % Hk)). A task source hands out task indices in the order the CTA runs
// them (first(), then next() until it returns -1, all CTA-uniform), tells which task next() will return
// (peek(), -1 if none) and is told when a task's record is complete (done()).
struct StridedTasks {
    int tau, ntask;
    __device__ __forceinline__ int first() { return tau < ntask ? tau : -1; }
    __device__ __forceinline__ int next() { tau += gridDim.x; return tau < ntask ? tau : -1; }
    __device__ __forceinline__ int peek() const { return tau + (int)gridDim.x < ntask ? tau + (int)gridDim.x : -1; }
    __device__ __forceinline__ void done(int, int) {}
};

// the two bf16 values of a 32-bit word as an fp32 pair (low half first)
__device__ __forceinline__ uint64_t f2_from_bf16x2(uint32_t u) { return f2_pack(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u)); }

// c = X Y for a 16 x K block of X (row-major, pitch lx) and a K x 8 block of Y (row-major, pitch ly), K a
// multiple of 8: m16n8k8 tf32 MMAs, operands rounded to tf32 (to nearest), fp32 accumulation; one warp. The
// inverse's result is rounded to fp16 before every use, so products at tf32 precision leave the layer's error
// where it is (a CPU emulation of the blocked inverse on the workloads' inputs: 4.22e-4 / 4.26e-4 against
// 4.21e-4 / 4.32e-4 for fp32 products, outputs / state). The k loop stays rolled: its chain is
// latency-bound either way, and the compact code keeps the caller's loop within the instruction caches.
__device__ __forceinline__ void mma_tf32_16x8(float (&c)[4], const float *X, int lx, const float *Y, int ly, int K,
                                              int lane) {
    const int g = lane >> 2, t = lane & 3;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 1
    for (int k0 = 0; k0 < K; k0 += 8) {
        const uint32_t a[4] = {tf32_bits(X[g * lx + k0 + t]), tf32_bits(X[(g + 8) * lx + k0 + t]),
                               tf32_bits(X[g * lx + k0 + t + 4]), tf32_bits(X[(g + 8) * lx + k0 + t + 4])};
        const uint32_t b[2] = {tf32_bits(Y[(k0 + t) * ly + g]), tf32_bits(Y[(k0 + t + 4) * ly + g])};
        mma_tf32(acc, a, b);
    }
#pragma unroll
    for (int f = 0; f < 4; ++f) c[f] = acc[f];
}
// The gates (g and beta, [rows][Hv] fp32) of rows [row0, row0 + n) into L2: the whole 16-byte granules
// inside those rows only, so that the prefetch stays within the rows the task reads.
__device__ __forceinline__ void prefetch_gates(const LaunchCommon &p, int64_t row0, int n) {
    const float *arr[2] = {p.g, p.beta};
#pragma unroll
    for (int q = 0; q < 2; ++q) {
        const uintptr_t lo = reinterpret_cast<uintptr_t>(arr[q] + row0 * p.Hv);
        const uintptr_t hi = reinterpret_cast<uintptr_t>(arr[q] + (row0 + n) * p.Hv);
        const uintptr_t s0 = (lo + 15) & ~uintptr_t(15), s1 = hi & ~uintptr_t(15);
        if (s1 > s0) bulk_prefetch_l2(reinterpret_cast<const void *>(s0), (uint32_t)(s1 - s0));
    }
}

// Task (blk, hk)'s input tiles and gates into L2, for a CTA's first task while it waits for earlier work.
// A prefetch only places lines in L2, the point of coherence, so a write that lands later still wins.
__device__ __forceinline__ void prefetch_task_inputs(const LaunchCommon &p, int blk, int hk) {
    const SessRef s = p.s[find_session(p, blk)];
    const int pos0 = (blk - s.blk0) * kBlock, row0 = (int)(s.row0 + pos0);
    tma_prefetch_2d(&p.tm_q, hk * up::D, row0);
    tma_prefetch_2d(&p.tm_k, hk * up::D, row0);
    for (int gi = 0; gi < p.G; ++gi) tma_prefetch_2d(&p.tm_v, (hk * p.G + gi) * up::D, row0);
    prefetch_gates(p, row0, min(kBlock, s.n - pos0));
}

// named barrier `id` over n threads (whole warps): bar_sync waits, bar_arrive only signals (its earlier
// shared-memory writes are visible to the threads that wait on the same barrier)
__device__ __forceinline__ void bar_sync(int id, int n) { asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ void bar_arrive(int id, int n) { asm volatile("bar.arrive %0, %1;\n" ::"r"(id), "r"(n) : "memory"); }
// the m16n8 C fragment c (times s) into a row-major block Z (pitch lz)
__device__ __forceinline__ void store_c16x8(float *Z, int lz, const float (&c)[4], float s, int lane) {
    const int g = lane >> 2, t = lane & 3;
    *reinterpret_cast<float2 *>(Z + g * lz + 2 * t) = make_float2(s * c[0], s * c[1]);
    *reinterpret_cast<float2 *>(Z + (g + 8) * lz + 2 * t) = make_float2(s * c[2], s * c[3]);
}

// 8 fp32 values -> bf16 hi and lo halves, packed for one 16-byte core-matrix row each
__device__ __forceinline__ void split8(const float *v, uint4 &hi, uint4 &lo) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) split_bf16x2(v[2 * q], v[2 * q + 1], h[q], l[q]);
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

// hi + lo of 8 bf16 pairs (one core-matrix row of each half)
__device__ __forceinline__ void join8(uint4 hi, uint4 lo, float *v) {
    const uint32_t h[4] = {hi.x, hi.y, hi.z, hi.w}, l[4] = {lo.x, lo.y, lo.z, lo.w};
#pragma unroll
    for (int q = 0; q < 4; ++q)   // packed pairs (the same bits as two scalar adds)
        f2_unpack(f2_add(f2_from_bf16x2(h[q]), f2_from_bf16x2(l[q])), v[2 * q], v[2 * q + 1]);
}

// Runs the tasks that `src` hands out, in order, on the operand plan at `sm` with control words `ctl` and
// 512 TMEM columns at `tmem` (allocated by the caller); every thread of the CTA (512) calls it. A task is
// one (64-token block, q/k head) with each of the head's G v-heads; the next head's or task's inputs are
// staged while the current head's inverse runs. Returns false if a bounded wait ran out (the error word is
// set, nothing is left in flight). The mbarriers are initialised on entry and invalidated on return, so
// the plan's memory may serve other uses between calls.
template <bool kAct, class Src>
__device__ __forceinline__ bool prologue_run(const LaunchCommon &p, int64_t ch, unsigned char *sm, UmmaCtl *ctl,
                                             uint32_t tmem, Src &src) {
    using namespace up;
    unsigned char *AQh = sm + OFF_AQH, *AQl = sm + OFF_AQL, *Bh = sm + OFF_BH;
    unsigned char *Ph = sm + OFF_PH, *TBh = sm + OFF_TBH, *ATh = sm + OFF_ATH;
    float *Af = reinterpret_cast<float *>(sm + OFF_AF), *Tf = reinterpret_cast<float *>(sm + OFF_TF);
    float *Mt = reinterpret_cast<float *>(sm + OFF_MT);
    float *gam = reinterpret_cast<float *>(sm + OFF_SMALL), *bet = gam + kBlock, *egv = bet + kBlock;
    uint64_t *bar = ctl->bar;
    __nv_bfloat16 *rawq = reinterpret_cast<__nv_bfloat16 *>(sm + OFF_RAW);
    __nv_bfloat16 *rawk = rawq + (kBlock + 3) * D, *rawv = rawk + (kBlock + 3) * D;
    __nv_bfloat16 *wq = reinterpret_cast<__nv_bfloat16 *>(sm + OFF_W), *wk = wq + 4 * D, *wv = wk + 4 * D;

    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    // the launch parameters used inside the task loop, read once (each later read of a field is a load)
    const int Hk = p.Hk, Hv = p.Hv, G = p.G, blk_lo = p.blk_lo, nblk = p.nblk;
    const bool block_major = p.task_block_major != 0;
    const int n_sess = p.n_sess;
    const long long wait_limit = p.wait_limit;
    const float *gate_g = p.g, *gate_beta = p.beta;
    const int64_t nq = (int64_t)Hk * D, nv = (int64_t)Hv * D;
    const __nv_bfloat16 *cw = static_cast<const __nv_bfloat16 *>(p.conv_w);
    struct Task { int blk, hk, pos0, n; int64_t row0, srow0; const void *conv0; };
    // the session of block blk: the last one that starts at or before it (a binary search in shared memory)
    const SessLite *sess = reinterpret_cast<const SessLite *>(sm + OFF_SESS);
    auto task_of = [&](int tau) {
        Task k;
        if (block_major) {
            k.blk = blk_lo + tau / Hk;
            k.hk = tau % Hk;
        } else {
            k.blk = blk_lo + tau % (nblk - blk_lo);
            k.hk = tau / (nblk - blk_lo);
        }
        int lo = 0;
        for (int hi = n_sess - 1; lo < hi;) {
            const int mid = (lo + hi + 1) >> 1;
            if (sess[mid].blk0 <= k.blk) lo = mid;
            else hi = mid - 1;
        }
        const SessLite ss = sess[lo];
        k.pos0 = (k.blk - ss.blk0) * kBlock;
        k.n = min(kBlock, ss.n - k.pos0);
        k.row0 = ss.row0 + k.pos0;
        k.srow0 = ss.row0;
        k.conv0 = ss.conv0;
        return k;
    };
    if (t == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        mbar_init_fence();
    }
    if (t < n_sess) {
        SessLite *w = reinterpret_cast<SessLite *>(sm + OFF_SESS) + t;
        w->row0 = p.s[t].row0;
        w->conv0 = p.s[t].conv0;
        w->n = p.s[t].n;
        w->blk0 = p.s[t].blk0;
    }
    __syncthreads();
    int tau = src.first();
    if (tau < 0) {
        if (t == 0) { mbar_inval(&bar[0]); mbar_inval(&bar[1]); }
        __syncthreads();
        return true;
    }
    Task cur = task_of(tau);
    int blk = cur.blk, hk = cur.hk, n = cur.n, ntau = -1;
    uint32_t in_phase = 0, mma_phase = 0;
    int in_pending = 0, mma_pending = 0;   // an issued copy group / MMA group not yet seen complete (CTA-uniform)

    // Stage rows pos0-3 .. pos0+63 of task k's q and k tiles (with_qk) and of v-head h's v tile, with their
    // conv weights: one tensor copy of the block's 64 rows per tile (rows past the inputs read as zero, rows
    // past n belong to other tokens and only reach masked results), issued by thread 256 with the byte count;
    // the three halo rows (from the inputs or, before a call's first token, from the conv state) and the
    // weights as single bulk copies, one per issuing thread (lanes 0 and 1 of warps 8-15). Every thread calls
    // it; the issuing threads are those that are idle while the inverse runs, where the next copies go out.
    struct Tile { __nv_bfloat16 *dst, *wdst; const CUtensorMap *map; const __nv_bfloat16 *x; int64_t ld, col0, chan0; };
    auto tile_of = [&](int q, const Task &k, int h) -> Tile {
        if (q == 0) return {rawq, wq, &p.tm_q, static_cast<const __nv_bfloat16 *>(p.xq), nq, (int64_t)k.hk * D, (int64_t)k.hk * D};
        if (q == 1)
            return {rawk, wk, &p.tm_k, static_cast<const __nv_bfloat16 *>(p.xk), nq, (int64_t)k.hk * D, nq + (int64_t)k.hk * D};
        return {rawv, wv, &p.tm_v, static_cast<const __nv_bfloat16 *>(p.xv), nv, (int64_t)h * D, 2 * nq + (int64_t)h * D};
    };
    auto stage = [&](const Task &k, int h, bool with_qk, bool skip) {
        if (skip) return;
        const int q0 = with_qk ? 0 : 2, ntile = 3 - q0;
        const int e = t >= 256 && lane < 2 ? ((t - 256) >> 5) + 8 * lane : 64;   // this thread's halo row or weights
        // the region was last read by generic loads (ordered by the barriers since): order them before the
        // async-proxy writes of the copies
        if (t == 256 || e < 4 * ntile) fence_proxy_async();
        if (t == 256) {
            mbar_arrive_expect_tx(&bar[0], (uint32_t)ntile * TILE_BYTES);
            for (int q = q0; q < 3; ++q) {
                const Tile tl = tile_of(q, k, h);
                tma_load_2d(tl.dst + 3 * D, tl.map, (int)tl.col0, (int)k.row0, &bar[0]);
            }
        }
        if (e < 4 * ntile) {
            const int r = e & 3;
            const Tile tl = tile_of(q0 + (e >> 2), k, h);
            if (r < 3) {
                const int pos = k.pos0 - 3 + r;
                const __nv_bfloat16 *src = pos < 0 ? static_cast<const __nv_bfloat16 *>(k.conv0) + (int64_t)(3 + pos) * ch + tl.chan0
                                                   : tl.x + (k.srow0 + pos) * tl.ld + tl.col0;
                bulk_g2s(tl.dst + r * D, src, RAW_ROW, &bar[0]);
            } else {
                bulk_g2s(tl.wdst, cw + tl.chan0 * 4, W_BYTES, &bar[0]);
            }
        }
    };
    // every thread waits; true when the phase completed for all of them (CTA-uniform)
    auto wait_in = [&]() {
        const bool ok = mbar_wait_bounded(&bar[0], in_phase, wait_limit);
        if (__syncthreads_or(!ok)) return false;
        in_phase ^= 1u;
        in_pending = 0;
        return true;
    };
    auto wait_mma = [&]() {
        const bool ok = mbar_wait_bounded(&bar[1], mma_phase, wait_limit);
        if (__syncthreads_or(!ok)) return false;
        mma_phase ^= 1u;
        mma_pending = 0;
        tc_fence_after();
        return true;
    };
    // bf16 hi/lo MMA group D (+)= A B over K (3 passes per 16-wide K-step), then a commit; thread 0 only.
    // The loop stays rolled (the issue is serial either way; compact code keeps the task loop in the
    // instruction caches).
    auto mma3 = [&](uint32_t d, uint64_t ah, uint64_t al, uint32_t astep, uint64_t bh, uint64_t bl, uint32_t bstep,
                    int K, uint32_t id) {
        tc_fence_after();
#pragma unroll 1
        for (int ks = 0; ks < K / 16; ++ks) {
            const uint64_t oa = (astep * ks) >> 4, ob = (bstep * ks) >> 4;
            umma_bf16(d, ah + oa, bh + ob, id, ks > 0);
            umma_bf16(d, ah + oa, bl + ob, id, 1);
            umma_bf16(d, al + oa, bh + ob, id, 1);
        }
        umma_commit(&bar[1]);
    };
    // single-pass fp16 MMA group D = A B over K, then a commit; thread 0 only
    auto mma1 = [&](uint32_t d, uint64_t a, uint32_t astep, uint64_t b, uint32_t bstep, int K, uint32_t id) {
        tc_fence_after();
#pragma unroll 1
        for (int ks = 0; ks < K / 16; ++ks) umma_bf16(d, a + ((astep * ks) >> 4), b + ((bstep * ks) >> 4), id, ks > 0);
        umma_commit(&bar[1]);
    };

    // Row-parallel conv of rows [r0, r0 + nr) of a staged tile: lane owns channels 4 lane .. 4 lane + 3,
    // four rows at a time; outputs go through emit(i0, y[4][4]). The taps run on channel pairs in packed
    // fp32 (oldest tap first: a product, then three fmas, per channel).
    auto conv_rows = [&](const __nv_bfloat16 *raw, const __nv_bfloat16 *wsm, int r0, int nr, auto &&emit) {
        uint64_t w2[2][4];   // [channel pair][tap]
        {
            const uint4 u0 = *reinterpret_cast<const uint4 *>(wsm + lane * 16);
            const uint4 u1 = *reinterpret_cast<const uint4 *>(wsm + lane * 16 + 8);
            const uint32_t ww[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};   // channel c: ww[2c], ww[2c + 1]
            float w[4][4];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                w[e >> 1][2 * (e & 1)] = __uint_as_float(ww[e] << 16);
                w[e >> 1][2 * (e & 1) + 1] = __uint_as_float(ww[e] & 0xFFFF0000u);
            }
#pragma unroll
            for (int q = 0; q < 2; ++q)
#pragma unroll
                for (int k = 0; k < 4; ++k) w2[q][k] = f2_pack(w[2 * q][k], w[2 * q + 1][k]);
        }
        for (int i0 = r0; i0 < r0 + nr; i0 += 4) {
            uint64_t x2[7][2];   // raw rows i0 .. i0+6 = block rows i0-3 .. i0+3, channel pairs
#pragma unroll
            for (int r = 0; r < 7; ++r) {
                const uint2 u = *reinterpret_cast<const uint2 *>(raw + (i0 + r) * D + lane * 4);
                x2[r][0] = f2_from_bf16x2(u.x);
                x2[r][1] = f2_from_bf16x2(u.y);
            }
            float y[4][4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    uint64_t a = f2_mul(w2[q][0], x2[u][q]);
                    a = f2_fma(w2[q][1], x2[u + 1][q], a);
                    a = f2_fma(w2[q][2], x2[u + 2][q], a);
                    a = f2_fma(w2[q][3], x2[u + 3][q], a);
                    f2_unpack(a, y[u][2 * q], y[u][2 * q + 1]);
                }
            if constexpr (kAct) {   // SiLU (a separate kernel instantiation, so the default one carries no code for it)
#pragma unroll
                for (int u = 0; u < 4; ++u)
#pragma unroll
                    for (int c = 0; c < 4; ++c) y[u][c] = y[u][c] / (1.0f + expf(-y[u][c]));
            }
            emit(i0, y);
        }
    };
    auto split4_store = [&](unsigned char *hi, unsigned char *lo, uint32_t off, const float (&v)[4]) {
        uint32_t h0, h1, l0, l1;
        split_bf16x2(v[0], v[1], h0, l0);
        split_bf16x2(v[2], v[3], h1, l1);
        *reinterpret_cast<uint2 *>(hi + off) = make_uint2(h0, h1);
        *reinterpret_cast<uint2 *>(lo + off) = make_uint2(l0, l1);
    };

    // beta v of the staged v-head (row-parallel conv, groups of 4 rows) into channels 128..255 of the B operand:
    // every warp takes the 4-row group `warp` (all), or, while thread 0 issues the Q K^T product, warps 1-15
    // take the 16 groups, warp 1 two of them (without_warp0)
    auto conv_v = [&](bool without_warp0) {
        if (without_warp0 && warp == 0) return;
        const int g0 = without_warp0 ? warp - 1 : warp, ng = without_warp0 && warp == 1 ? 2 : 1;
        auto emit = [&](int i0, float (&y)[4][4]) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u;
                float v[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) v[c] = i < n ? bet[i] * y[u][c] : 0.f;
                *reinterpret_cast<uint2 *>(Bh + mnmajor_bf16_offset(128 + 4 * lane, i, B_LBO, B_SBO)) =
                    make_uint2(f2_to_h2(v[0], v[1]), f2_to_h2(v[2], v[3]));
            }
        };
#pragma unroll 1
        for (int k = 0; k < ng; ++k) conv_rows(rawv, wv, 4 * (k == 0 ? g0 : 15), 4, emit);   // group 15 to warp 1
    };
    // channels 0..127 of the B operand: beta e^gamma k_hat (from the hi/lo rows), 1024 groups of 8 channels,
    // over every thread, or (for the first v-head, where warp 1 takes two conv groups and warp 0 joins after
    // issuing the Q K^T product) over every thread but warp 1's
    auto b_khat = [&](bool without_warp1) {
        if (without_warp1 && warp == 1) return;
        // (warp 0 ranks last there, so that the 64 threads with a third group are in warps 2 and 3)
        const int r0 = !without_warp1 ? t : (warp == 0 ? kUmmaPrepThreads - 64 + lane : t - 64);
        const int nr = without_warp1 ? kUmmaPrepThreads - 32 : kUmmaPrepThreads;
        for (int e = r0; e < 64 * 16; e += nr) {
            const int j = e & 63, cg = e >> 6;
            const uint32_t o = kmajor_bf16_offset(64 + j, 8 * cg, AQ_LBO, AQ_SBO);
            float v[8];
            join8(*reinterpret_cast<const uint4 *>(AQh + o), *reinterpret_cast<const uint4 *>(AQl + o), v);
            const float sc = bet[j] * egv[j];
#pragma unroll
            for (int c = 0; c < 8; c += 2) f2_unpack(f2_mul(f2_pack(v[c], v[c + 1]), f2_pack(sc, sc)), v[c], v[c + 1]);
            *reinterpret_cast<uint4 *>(Bh + mnmajor_bf16_offset(8 * cg, j, B_LBO, B_SBO)) = f8_to_h8(v);
        }
    };

    stage(cur, hk * G, true, p.debug_skip_first_copy == 2);   // 1. the first task's tiles
    in_pending = 1;
    // gamma (inclusive scan of g over the block), beta and e^gamma of v-head h, by warps 8 and 9 alone: warp 9
    // adds the total of rows 0..31 itself, so no barrier is needed. The loads are issued early (for the
    // next head or task, while the inverse of the current one runs) and the scan run later.
    const int jg = t - 256;
    struct Gv { float g, b, lo; };
    auto gates_load = [&](const Task &k, int h) {
        Gv r{0.f, 0.f, 0.f};
        if (jg < 0 || jg >= kBlock) return r;
        if (jg < k.n) {
            r.g = gate_g[(k.row0 + jg) * Hv + h];
            r.b = gate_beta[(k.row0 + jg) * Hv + h];
        }
        if (jg >= 32 && lane < k.n) r.lo = gate_g[(k.row0 + lane) * Hv + h];
        return r;
    };
    auto gates_store = [&](Gv r) {
        if (jg < 0 || jg >= kBlock) return;
        float sv = r.g, lo = r.lo;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, sv, o);
            if (lane >= o) sv += y;
        }
        if (jg >= 32) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) lo += __shfl_xor_sync(0xffffffffu, lo, o);
            sv += lo;
        }
        gam[jg] = sv;
        bet[jg] = r.b;
        egv[jg] = expf(sv);
    };
    gates_store(gates_load(cur, hk * G));
    Gv gnext{0.f, 0.f, 0.f}, ghead{0.f, 0.f, 0.f};
    bool ok = true;
    for (;;) {   // tasks
    ok = wait_in();

    if (ok) {
        // 2. conv + L2 norm of q (warps 0-7) and k (warps 8-15), 8 rows per warp -> bf16 hi/lo rows of [q_hat; k_hat]
        const int which = warp >> 3;
        const float qs = which ? 1.f : p.q_scale;
        conv_rows(which ? rawk : rawq, which ? wk : wq, 8 * (warp & 7), 8, [&](int i0, float (&y)[4][4]) {
            float ss[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                ss[u] = 0.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) ss[u] = fmaf(y[u][c], y[u][c], ss[u]);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                for (int u = 0; u < 4; ++u) ss[u] += __shfl_xor_sync(0xffffffffu, ss[u], o);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u;
                const float scale = qs * rsqrtf(ss[u] + p.eps);
                float v[4];
#pragma unroll
                for (int c = 0; c < 4; ++c) v[c] = i < n ? y[u][c] * scale : 0.f;
                split4_store(AQh, AQl, kmajor_bf16_offset(64 * which + i, 4 * lane, AQ_LBO, AQ_SBO), v);
            }
        });
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();
        // 3. [Q K^T; K K^T] = [q_hat; k_hat] k_hat^T into TMEM columns 0..63 (the first v-head's B operand is
        //    built on warps 1-15 meanwhile)
        if (t == 0)
            mma3(tmem, umma_smem_desc(AQh, AQ_LBO, AQ_SBO), umma_smem_desc(AQl, AQ_LBO, AQ_SBO), 2 * AQ_LBO,
                 umma_smem_desc(AQh + 8 * AQ_SBO, AQ_LBO, AQ_SBO), umma_smem_desc(AQl + 8 * AQ_SBO, AQ_LBO, AQ_SBO),
                 2 * AQ_LBO, D, umma_idesc_bf16(128, 64, 0, 0));
        mma_pending = 1;
    }

    // 4. each v-head of the group
    for (int gi = 0; ok && gi < G; ++gi) {
        const int h = hk * G + gi;
        if (gi > 0) {   // this head's v tile was staged while the previous head's inverse ran
            gates_store(ghead);
            if (!(ok = wait_in())) break;
        }
        unsigned char *rec = reinterpret_cast<unsigned char *>(p.ws_wu) + ((int64_t)blk * Hv + h) * rec16::kBytes;
        // K_tilde^T as the fp16 MN-major A operand (d_k x 64 tokens): a 16-byte core row is 8 channels of one
        // token's e^{gamma_63 - gamma_j} k_hat, so each comes from one row chunk of k_hat; half `part` of the
        // 1,024 chunks, by warps 1-15 (warp 0 issues the MMAs), consecutive threads on consecutive record
        // bytes; e^{gamma_63} with the first half
        auto kt_record = [&](int part) {
            if (warp == 0) return;
            constexpr int HALF = 512;
            const float gl = gam[kBlock - 1];
            for (int e = HALF * part + t - 32; e < HALF * (part + 1); e += kUmmaPrepThreads - 32) {
                const int j = 8 * (e >> 7) + (e & 7), dg = (e >> 3) & 15;
                const uint32_t o = kmajor_bf16_offset(kBlock + j, 8 * dg, AQ_LBO, AQ_SBO);
                float v[8];
                join8(*reinterpret_cast<const uint4 *>(AQh + o), *reinterpret_cast<const uint4 *>(AQl + o), v);
                const float dec = __expf(gl - gam[j]);
#pragma unroll
                for (int c = 0; c < 8; c += 2) f2_unpack(f2_mul(f2_pack(v[c], v[c + 1]), f2_pack(dec, dec)), v[c], v[c + 1]);
                *reinterpret_cast<uint4 *>(rec + rec16::kt(8 * dg, j)) = f8_to_h8(v);
            }
            if (part == 0 && t == 32) *reinterpret_cast<float *>(rec + rec16::kEg) = expf(gl);
        };

        // 5. B operand, MN-major: channels 128..255 = beta v, channels 0..127 = beta e^gamma k_hat; for the
        //    first v-head on warps 1-15 while thread 0 issues the Q K^T product
        conv_v(gi == 0);
        b_khat(gi == 0);
        fence_proxy_async();
        if (gi == 0) {
            if (!(ok = wait_mma())) break;   // Q K^T / K K^T landed in TMEM
        } else {
            __syncthreads();
        }

        // 6. from TMEM: P (rows 0..63 -> bf16 hi/lo K-major) and A (rows 64..127 -> fp32)
        {
            const int q = warp & 3, cp = warp >> 2, R = 32 * q + lane, j0 = 16 * cp;
            uint32_t r[16];
            tmem_ld16_nowait(tmem + ((uint32_t)(32 * q) << 16) + j0, r);
            float dec[16];   // e^{gamma_i - gamma_j}, while the load is in flight
            {
                const float gr = gam[R < kBlock ? R : R - kBlock];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) dec[jj] = __expf(gr - gam[j0 + jj]);
            }
            tmem_wait_ld(r);
            float v[16];
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) v[jj] = __uint_as_float(r[jj]);
            if (R < kBlock) {
                const int i = R;
                float pv[16];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) pv[jj] = (j0 + jj) <= i ? v[jj] * dec[jj] : 0.f;
                *reinterpret_cast<uint4 *>(Ph + kmajor_bf16_offset(i, j0, K64_LBO, K64_SBO)) = f8_to_h8(pv);
                *reinterpret_cast<uint4 *>(Ph + kmajor_bf16_offset(i, j0 + 8, K64_LBO, K64_SBO)) = f8_to_h8(pv + 8);
            } else {
                const int i = R - kBlock;
                float av[16];
#pragma unroll
                for (int jj = 0; jj < 16; ++jj) av[jj] = (j0 + jj) < i ? bet[i] * dec[jj] * v[jj] : 0.f;
#pragma unroll
                for (int c = 0; c < 16; c += 4)
                    *reinterpret_cast<float4 *>(Af + i * LT + j0 + c) = make_float4(av[c], av[c + 1], av[c + 2], av[c + 3]);
            }
        }
        tc_fence_before();
        __syncthreads();

        // the next v-head's v tile, or the next task's inputs: every raw tile and weight of this head has been
        // read, so their region takes the next copies now, a whole head's work ahead of their use. Warps 8-15,
        // idle in the inverse, work out the next task (and leave it in shared memory for the other warps),
        // issue the copies and load the gates (which go to shared memory once this head's record is written).
        const bool next_head = gi + 1 < G;
        const int ptau = next_head ? -1 : src.peek();   // the task that next() returns at the end of this one
        const bool stage_next = next_head || ptau >= 0;
        if (stage_next) in_pending = 1;

        // 7. T = (I + A)^{-1} (unit lower triangular) in fp32, two levels of 2x2 blocking, products as
        //    tf32 MMAs, one 16 x 8 tile per warp:
        //    (a) diagonal 16x16 blocks D_b by substitution, one column per thread (warp 0: D_0, D_1; warp 1:
        //        D_2, D_3); warps 8-15 zero the blocks above the diagonal, then issue the copies above;
        //    (b) warps 0-3 (block pair (b + 1, b), column tile nt): T_10 = -D_1 (A_10 D_0), T_32 = -D_3 (A_32 D_2);
        //    (c) warps 0-7 (row tile mt, column tile nt): X = A[32:64, 0:32] T[0:32, 0:32], then
        //        T[32:64, 0:32] = -T[32:64, 32:64] X.
        //    Products skip the zero blocks of T, whose writes need only be done by the CTA barrier after (c).
        //    Named barriers order the levels: 1 (warps 0-3), 2 (warps 0-7), 3 + nt (X tile (0, nt) from warp
        //    nt to warp 4 + nt).
        constexpr int LM = 24, LX = 40;
        float *Xs = reinterpret_cast<float *>(TBh);   // 32 x LX scratch (the T operand regions are written later)
        if (t < kBlock) {
            const int d = t >> 4, c = t & 15;
            const float *Ad = Af + 16 * d * LT + 16 * d;
            // right-looking: once x_j is final, every later row takes its term (x_j = 0 for j < c adds
            // nothing), so the dependent chain is one fma per row
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) x[i] = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const float xj = j < c ? 0.f : (j == c ? 1.f : x[j]);
                x[j] = xj;
#pragma unroll
                for (int i = j + 1; i < 16; ++i) x[i] = fmaf(-Ad[i * LT + j], xj, x[i]);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) Tf[(16 * d + i) * LT + 16 * d + c] = x[i];
        } else if (t >= 256) {
            for (int e = t - 256; e < 6 * 64; e += kUmmaPrepThreads - 256) {   // 6 blocks x 16 rows x 4 float4
                const int bi = e >> 6, r = (e >> 2) & 15, c4 = e & 3;
                const int ib = bi < 3 ? 0 : (bi < 5 ? 1 : 2), jb = bi < 3 ? bi + 1 : (bi < 5 ? bi - 1 : 3);
                *reinterpret_cast<float4 *>(Tf + (16 * ib + r) * LT + 16 * jb + 4 * c4) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            if (stage_next) {
                const Task k = next_head ? cur : task_of(ptau);
                const int hs = next_head ? h + 1 : k.hk * G;
                if (!next_head && t == 256) *reinterpret_cast<Task *>(sm + OFF_NEXT) = k;
                stage(k, hs, !next_head, false);
                const Gv gv = gates_load(k, hs);
                if (next_head) ghead = gv;
                else gnext = gv;
            }
        }
        if (warp < 4) {   // (b)
            bar_sync(1, 128);
            const int b = 2 * (warp >> 1), nt = warp & 1;
            float *M = Mt + (warp >> 1) * 16 * LM;
            float cc[4];
            mma_tf32_16x8(cc, Af + 16 * (b + 1) * LT + 16 * b, LT, Tf + 16 * b * LT + 16 * b + 8 * nt, LT, 16, lane);
            store_c16x8(M + 8 * nt, LM, cc, 1.f, lane);
            __syncwarp();
            mma_tf32_16x8(cc, Tf + 16 * (b + 1) * LT + 16 * (b + 1), LT, M + 8 * nt, LM, 16, lane);
            store_c16x8(Tf + 16 * (b + 1) * LT + 16 * b + 8 * nt, LT, cc, -1.f, lane);
        }
        if (warp < 8) {   // (c)
            bar_sync(2, 256);
            const int nt = warp & 3, mt = warp >> 2;
            float cc[4];
            // T[0:16, 16:32] = 0: column tiles 2 and 3 of T[0:32, 0:32] need only its rows 16..31
            const int k0 = nt < 2 ? 0 : 16;
            mma_tf32_16x8(cc, Af + (32 + 16 * mt) * LT + k0, LT, Tf + k0 * LT + 8 * nt, LT, 32 - k0, lane);
            store_c16x8(Xs + 16 * mt * LX + 8 * nt, LX, cc, 1.f, lane);
            // T[32:48, 48:64] = 0: row tile 0 needs only X rows 0..15 (its own tile), row tile 1 all 32
            if (mt == 0) {
                bar_arrive(3 + nt, 64);
                __syncwarp();
            } else {
                bar_sync(3 + nt, 64);
            }
            mma_tf32_16x8(cc, Tf + (32 + 16 * mt) * LT + 32, LT, Xs + 8 * nt, LX, 16 + 16 * mt, lane);
            store_c16x8(Tf + (32 + 16 * mt) * LT + 8 * nt, LT, cc, -1.f, lane);
        }
        __syncthreads();
        //    T as fp16: rows 0..63 of [T; P T] (K-major, written over A and T) and the B operand of
        //    P T (MN-major)
        {
            const int i = t & 63, kg = t >> 6;
            float v[8];
            const float4 a = *reinterpret_cast<const float4 *>(Tf + i * LT + 8 * kg);
            const float4 b = *reinterpret_cast<const float4 *>(Tf + i * LT + 8 * kg + 4);
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
            __syncthreads();   // every row of T is read before the first write over it
            const uint4 th = f8_to_h8(v);
            *reinterpret_cast<uint4 *>(ATh + kmajor_bf16_offset(i, 8 * kg, K64_LBO, K64_SBO)) = th;
            *reinterpret_cast<uint4 *>(TBh + mnmajor_bf16_offset(8 * kg, i, K64_LBO, K64_SBO)) = th;
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();

        // 8. P T into TMEM columns 64..127; meanwhile the first half of the K_tilde^T record
        if (t == 0)
            mma1(tmem + 64, umma_smem_desc(Ph, K64_LBO, K64_SBO), 2 * K64_LBO, umma_smem_desc(TBh, K64_LBO, K64_SBO),
                 2 * K64_LBO, kBlock, umma_idesc_f16(128, 64, 0, 1));
        mma_pending = 1;
        kt_record(0);   // the first half of K_tilde^T while the product runs, the second under the next one
        if (!(ok = wait_mma())) break;

        // 9. P T (lanes 0..63; warps 0,1,4,5,8,9,12,13, 16 columns each) -> rows 64..127 of [T; P T]
        if ((warp & 3) < 2) {
            const int i = 32 * (warp & 3) + lane, c0 = 16 * (warp >> 2);
            float v[16];
            tmem_ld16(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 64 + c0, v);
            *reinterpret_cast<uint4 *>(ATh + kmajor_bf16_offset(kBlock + i, c0, K64_LBO, K64_SBO)) = f8_to_h8(v);
            *reinterpret_cast<uint4 *>(ATh + kmajor_bf16_offset(kBlock + i, c0 + 8, K64_LBO, K64_SBO)) = f8_to_h8(v + 8);
        }
        fence_proxy_async();
        tc_fence_before();
        __syncthreads();

        // 10. [W U; P W P U] = [T; P T] [beta e^gamma k_hat | beta v] into TMEM columns 256..511
        if (t == 0)
            mma1(tmem + 256, umma_smem_desc(ATh, K64_LBO, K64_SBO), 2 * K64_LBO, umma_smem_desc(Bh, B_LBO, B_SBO),
                 2 * B_LBO, kBlock, umma_idesc_f16(128, 256, 0, 1));
        mma_pending = 1;
        kt_record(1);
        if (!(ok = wait_mma())) break;

        // 11. the record, every warp (lanes 32 (warp % 4) .., the 16-column chunks warp / 4 + 4 j, j = 0..3: two of
        //     [W; P W] and two of [U; P U], so that every warp has the same share of the costlier first kind),
        //     in fp16: W rows -> rows 0..63 of the [W; Qe] operand; P W rows -> Qe = e^gamma q_hat - P W, rows
        //     64..127; U rows -> U; P U rows -> O_intra
        {
            const int R = 32 * (warp & 3) + lane, cp = warp >> 2;
            const bool top = R < kBlock;
            const int i = top ? R : R - kBlock;
            const uint32_t tb = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 256;
#pragma unroll 1
            for (int cc = 0; cc < 4; ++cc) {
                const int c0 = 16 * (cp + 4 * cc);
                float v[16];
                tmem_ld16(tb + c0, v);
                uint32_t off, step;
                if (c0 < D) {
                    if (!top) {
                        float qh[16];
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const uint32_t o = kmajor_bf16_offset(i, c0 + 8 * hh, AQ_LBO, AQ_SBO);
                            join8(*reinterpret_cast<const uint4 *>(AQh + o), *reinterpret_cast<const uint4 *>(AQl + o), qh + 8 * hh);
                        }
                        const float e = egv[i];
#pragma unroll
                        for (int c = 0; c < 16; ++c) v[c] = e * qh[c] - v[c];
                    }
                    off = rec16::wq(R, c0);
                    step = 128;   // the next 8 columns: the core matrix adjacent along K
                } else {
                    off = (top ? rec16::kU : rec16::kO) + rec16::uo(i, c0 - D);
                    step = 1024;  // the next 8 columns
                }
                *reinterpret_cast<uint4 *>(rec + off) = f8_to_h8(v);
                *reinterpret_cast<uint4 *>(rec + off + step) = f8_to_h8(v + 8);
            }
        }
        tc_fence_before();
        __syncthreads();   // TMEM columns and every operand region are free for the next v-head
    }
    if (!ok) break;
    src.done(blk, hk);   // the task's record is complete
    if ((ntau = src.next()) < 0) break;
    tau = ntau;
    cur = *reinterpret_cast<const Task *>(sm + OFF_NEXT);
    blk = cur.blk; hk = cur.hk; n = cur.n;
    gates_store(gnext);
    }   // tasks

    if (!ok) {   // a bounded wait ran out: record it and wait (bounded) for what is still in flight
        if (t == 0) {
            atomicOr(p.err, 1u);
            if (in_pending && p.debug_skip_first_copy != 2) mbar_wait_bounded(&bar[0], in_phase, wait_limit);
            if (mma_pending) mbar_wait_bounded(&bar[1], mma_phase, wait_limit);
        }
        tc_fence_before();
        __syncthreads();
    }
    tc_fence_after();
    if (t == 0) { mbar_inval(&bar[0]); mbar_inval(&bar[1]); }
    __syncthreads();
    return ok;
}


}  // namespace gdn
