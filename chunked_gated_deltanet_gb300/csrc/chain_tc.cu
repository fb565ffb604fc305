// Sequential state pass and outputs on tensor cores (bf16-input path): one CTA
// per (session, v-head, 16-column slice of d_v), 8 warps, walking the
// session's 64-token blocks strictly in position order. Per block:
//   Z = [W; Qe] S^T                  (128 x 16; warp w owns rows 16w..16w+15)
//   U' = U - Z[0:64],  O = Z[64:128] + O_intra   (outputs written here)
//   S^T <- e^{gamma_63} S^T + K_tilde^T U'        (warp w owns state rows 16w..16w+15)
// The fp32 state lives in the registers of the warps that own its rows (in
// m16n8 accumulator layout); shared memory holds its tf32 copy, the B operand
// of the next block's first product. Operands are tf32 (rounded by the
// prologue, or here for U'), accumulation is fp32. The prologue stores each
// block's operands in fragment order, so a block is five contiguous bulk
// copies (TMA), issued by one thread into a two-stage buffer and completed on
// an mbarrier; block b+1 loads while block b computes. Every wait on an
// mbarrier is bounded: on timeout the CTA records GDN_ERR_TIMEOUT in the
// device error word, waits (bounded) for its copies in flight, and returns.
// The CTA also commits its share of the session's conv state.
#include "common.cuh"
#include "mma.cuh"

__device__ unsigned int g_gdn_device_error;

namespace gdn {

// Shared-memory plan of a CTA with DS state columns. With 16 columns both operand sets of a block (A of
// the first product, [W; Qe], and of the second, K_tilde^T, with the U and O_intra slices) are double
// buffered. With 32 columns that does not fit: the K_tilde^T part stays double buffered and [W; Qe] has
// one buffer, refilled for the next block while the second product runs.
template <int D, int DS>
struct ChainPlan {
    static constexpr bool kSplit = DS > kSliceCols;
    static constexpr int SP = DS + 8;          // tf32 S^T and U' rows (B fragments): banks 8t + g, distinct
    static constexpr int WQF = 2 * kBlock * D; // [W; Qe] fragments
    static constexpr int KTF = kBlock * D;     // K_tilde^T fragments
    static constexpr int UF = kBlock * DS;     // U (or O_intra) fragments of the CTA's columns
    static constexpr int KSTAGE = KTF + 2 * UF + 4;                        // K_tilde^T, U, O_intra, e^{gamma_63}
    static constexpr int STAGE = kSplit ? KSTAGE : WQF + KSTAGE;           // one double-buffered stage
    static constexpr int WQBUF = kSplit ? WQF : 0;                         // the single [W; Qe] buffer
    static constexpr size_t bytes() {
        return sizeof(float) * (2 * STAGE + WQBUF + D * SP + kBlock * SP) + 4 * sizeof(uint64_t);
    }
};

template <int D, int DS>
__global__ void __launch_bounds__(kThreads, 1) chain_tc_kernel(const LaunchCommon p, int64_t ch) {
    extern __shared__ __align__(16) float smem[];
    using P = ChainPlan<D, DS>;
    constexpr int NT = DS / 8, SP = P::SP, WQF = P::WQF, KTF = P::KTF, UF = P::UF, STAGE = P::STAGE;
    constexpr bool kSplit = P::kSplit;
    static_assert(D == 128 || D == 64, "head dim");
    static_assert(DS == 16 || DS == 32, "slice width");
    float *wqbuf = smem + 2 * STAGE;           // [W; Qe] of the current block (split plan only)
    float *St = wqbuf + P::WQBUF;              // [D][SP]   tf32 copy of the state slice
    float *Ups = St + D * SP;                  // [64][SP]  tf32 U'
    uint64_t *bar = reinterpret_cast<uint64_t *>(Ups + kBlock * SP);   // [0..1] stages, [2] [W; Qe] buffer
    // block b's operands: A of the first product, then K_tilde^T, U, O_intra, e^{gamma_63}
    auto wq_of = [&](int b) -> const float * { return kSplit ? wqbuf : smem + (b & 1) * STAGE; };
    auto kt_of = [&](int b) -> const float * { return smem + (b & 1) * STAGE + (kSplit ? 0 : WQF); };

    constexpr int nsl = D / DS;
    const int sl = blockIdx.x % nsl;
    const int h = (blockIdx.x / nsl) % p.Hv;
    const int si = blockIdx.x / (nsl * p.Hv);
    const SessRef s = p.s[si];
    const int c0 = sl * DS, t = threadIdx.x, warp = t >> 5, lane = t & 31, g8 = lane >> 2, t4 = lane & 3;
    const int Hv = p.Hv;
    const int nb = (s.n + kBlock - 1) / kBlock;
    const int64_t RF = rec_floats(D);
    const bool owner = 16 * warp < D;          // this warp owns state rows 16w..16w+15
    const int m0 = 16 * warp + g8;

    // conv-state commit: the raw inputs at the session's last three processed positions
    {
        const int ncta = Hv * nsl, j = h * nsl + sl;
        const int64_t per = (ch + ncta - 1) / ncta, chan = j * per + t;
        if (t < per && chan < ch && s.n > 0) {
            const int64_t nq = (int64_t)p.Hk * D, nv = (int64_t)Hv * D;
            const __nv_bfloat16 *x;
            int64_t col, ld;
            if (chan < nq) { x = static_cast<const __nv_bfloat16 *>(p.xq); col = chan; ld = nq; }
            else if (chan < 2 * nq) { x = static_cast<const __nv_bfloat16 *>(p.xk); col = chan - nq; ld = nq; }
            else { x = static_cast<const __nv_bfloat16 *>(p.xv); col = chan - 2 * nq; ld = nv; }
            __nv_bfloat16 *cs = static_cast<__nv_bfloat16 *>(s.conv);
            const __nv_bfloat16 *cs0 = static_cast<const __nv_bfloat16 *>(s.conv0);
            const __nv_bfloat16 o0 = cs0[chan], o1 = cs0[ch + chan], o2 = cs0[2 * ch + chan];
            __nv_bfloat16 nw[3];
#pragma unroll
            for (int r = 0; r < 3; ++r) {
                const int pos = s.n - 3 + r;
                nw[r] = pos >= 0 ? x[(s.row0 + pos) * ld + col] : (pos == -3 ? o0 : (pos == -2 ? o1 : o2));
            }
#pragma unroll
            for (int r = 0; r < 3; ++r) cs[r * ch + chan] = nw[r];
            if (s.conv_cap) {
                __nv_bfloat16 *cc = static_cast<__nv_bfloat16 *>(s.conv_cap);
#pragma unroll
                for (int r = 0; r < 3; ++r) cc[r * ch + chan] = nw[r];
            }
        }
    }

    // block b's operands -> stage b & 1 (thread 0 only): with the 16-column plan all of them, with the
    // split plan the K_tilde^T part ([W; Qe] goes through issue_wq)
    constexpr int CHUNK = 4096;   // floats per bulk copy (16 KB)
    static_assert(WQF % CHUNK == 0 && KTF % CHUNK == 0, "operand blocks are whole numbers of chunks");
    auto issue = [&](int b) {
        float *buf = smem + (b & 1) * STAGE;
        const float *r = p.ws_wu + ((int64_t)(s.blk0 + b) * Hv + h) * RF;
        uint64_t *br = &bar[b & 1];
        if (b == 0 && p.debug_skip_first_copy == 1) return;   // test hook: leave the barrier pending
        fence_proxy_async();
        mbar_arrive_expect_tx(br, (uint32_t)sizeof(float) * STAGE);
        const int first = kSplit ? WQF / CHUNK : 0;           // the split plan skips [W; Qe]
#pragma unroll
        for (int q = first; q < (WQF + KTF) / CHUNK; ++q)
            bulk_g2s(buf + (q - first) * CHUNK, r + q * CHUNK, sizeof(float) * CHUNK, br);
        float *u = buf + STAGE - 2 * UF - 4;
        bulk_g2s(u, r + 192 * D + sl * UF, sizeof(float) * UF, br);
        bulk_g2s(u + UF, r + 256 * D + sl * UF, sizeof(float) * UF, br);
        bulk_g2s(u + 2 * UF, r + 320 * D, 16, br);
    };
    auto issue_wq = [&](int b) {   // split plan: [W; Qe] of block b into its single buffer
        const float *r = p.ws_wu + ((int64_t)(s.blk0 + b) * Hv + h) * RF;
        fence_proxy_async();
        mbar_arrive_expect_tx(&bar[2], (uint32_t)sizeof(float) * WQF);
#pragma unroll
        for (int q = 0; q < WQF / CHUNK; ++q) bulk_g2s(wqbuf + q * CHUNK, r + q * CHUNK, sizeof(float) * CHUNK, &bar[2]);
    };

    // state rows in registers (fp32), tf32 copy in shared memory
    float *Sg = s.S + (int64_t)h * D * D;
    const float *Sg0 = s.S0 + (int64_t)h * D * D;   // the starting state (the session's own, or a prefix's)
    float st[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int c = 8 * nt + 2 * t4;
        if (owner) {
            st[nt][0] = Sg0[(int64_t)m0 * D + c0 + c];
            st[nt][1] = Sg0[(int64_t)m0 * D + c0 + c + 1];
            st[nt][2] = Sg0[(int64_t)(m0 + 8) * D + c0 + c];
            st[nt][3] = Sg0[(int64_t)(m0 + 8) * D + c0 + c + 1];
            St[m0 * SP + c] = tf32_round(st[nt][0]);
            St[m0 * SP + c + 1] = tf32_round(st[nt][1]);
            St[(m0 + 8) * SP + c] = tf32_round(st[nt][2]);
            St[(m0 + 8) * SP + c + 1] = tf32_round(st[nt][3]);
        } else {
            st[nt][0] = st[nt][1] = st[nt][2] = st[nt][3] = 0.f;
        }
    }
    if (t == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        mbar_init(&bar[2], 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (t == 0 && nb > 0) {
        issue(0);
        if constexpr (kSplit) issue_wq(0);
    }

    int timed_out = 0;
    for (int b = 0; b < nb; ++b) {
        const float *wq = wq_of(b), *kt = kt_of(b), *uo0 = kt + KTF;
        if (t == 0 && b + 1 < nb) issue(b + 1);   // the other stage was released at the end of step b-1
        // every thread acquires the stage itself; a timeout is acted on at the end of the step
        if (!mbar_wait_bounded(&bar[b & 1], (b >> 1) & 1, p.wait_limit)) timed_out = b + 1;
        if constexpr (kSplit)
            if (!mbar_wait_bounded(&bar[2], b & 1, p.wait_limit)) timed_out = b + 1;

        // Z = [W; Qe] S^T, four partial accumulators per n-tile (k-step mod 4)
        float acc[4][NT][4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int f = 0; f < 4; ++f) acc[j][nt][f] = 0.f;
        {
            const float4 *wa = reinterpret_cast<const float4 *>(wq) + (warp * (D / 8)) * 32 + lane;
#pragma unroll
            for (int ks = 0; ks < D / 8; ++ks) {
                const float4 av = wa[ks * 32];
                const uint32_t a[4] = {__float_as_uint(av.x), __float_as_uint(av.y), __float_as_uint(av.z),
                                       __float_as_uint(av.w)};
                const int k0 = 8 * ks;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint32_t bb[2] = {__float_as_uint(St[(k0 + t4) * SP + 8 * nt + g8]),
                                            __float_as_uint(St[(k0 + t4 + 4) * SP + 8 * nt + g8])};
                    mma_tf32(acc[ks & 3][nt], a, bb);
                }
            }
        }
        // U' (warps 0-3) and outputs (warps 4-7); C fragments match the stored order
        {
            const int nrow = min(kBlock, s.n - b * kBlock);
            const int w4 = warp & 3;
            const float4 *uo = reinterpret_cast<const float4 *>(uo0 + (warp < 4 ? 0 : UF));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                // fragments are stored by 16-column slice: [slice][m-tile][n-tile of 8][lane][4]
                const float4 u = uo[(((nt >> 1) * 4 + w4) * 2 + (nt & 1)) * 32 + lane];
                float z[4];
#pragma unroll
                for (int f = 0; f < 4; ++f) z[f] = (acc[0][nt][f] + acc[1][nt][f]) + (acc[2][nt][f] + acc[3][nt][f]);
                const int c = 8 * nt + 2 * t4, i = 16 * w4 + g8;
                if (warp < 4) {
                    Ups[i * SP + c] = tf32_round(u.x - z[0]);
                    Ups[i * SP + c + 1] = tf32_round(u.y - z[1]);
                    Ups[(i + 8) * SP + c] = tf32_round(u.z - z[2]);
                    Ups[(i + 8) * SP + c + 1] = tf32_round(u.w - z[3]);
                } else {
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int ii = i + 8 * hh;
                        if (ii >= nrow) continue;
                        const float o0 = z[2 * hh] + (hh ? u.z : u.x), o1 = z[2 * hh + 1] + (hh ? u.w : u.y);
                        const int64_t oi = ((s.row0 + (int64_t)b * kBlock + ii) * Hv + h) * D + c0 + c;
                        if (p.out_bf16)
                            *reinterpret_cast<__nv_bfloat162 *>(static_cast<__nv_bfloat16 *>(p.out) + oi) =
                                __floats2bfloat162_rn(o0, o1);
                        else
                            *reinterpret_cast<float2 *>(static_cast<float *>(p.out) + oi) = make_float2(o0, o1);
                    }
                }
            }
        }
        __syncthreads();  // (B) U' complete; every read of the tf32 state copy and of [W; Qe] done
        if constexpr (kSplit)
            if (t == 0 && b + 1 < nb) issue_wq(b + 1);   // refilled while the second product runs
        // S^T <- e^{gamma_63} S^T + K_tilde^T U' on the owner warps' registers
        if (owner) {
            const float e = uo0[2 * UF];
            float cx[3][NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int f = 0; f < 4; ++f) {
                    st[nt][f] *= e;
                    cx[0][nt][f] = cx[1][nt][f] = cx[2][nt][f] = 0.f;
                }
            const float4 *ka = reinterpret_cast<const float4 *>(kt) + (warp * 8) * 32 + lane;
#pragma unroll
            for (int ks = 0; ks < kBlock / 8; ++ks) {
                const float4 av = ka[ks * 32];
                const uint32_t a[4] = {__float_as_uint(av.x), __float_as_uint(av.y), __float_as_uint(av.z),
                                       __float_as_uint(av.w)};
                const int k0 = 8 * ks;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint32_t bb[2] = {__float_as_uint(Ups[(k0 + t4) * SP + 8 * nt + g8]),
                                            __float_as_uint(Ups[(k0 + t4 + 4) * SP + 8 * nt + g8])};
                    mma_tf32((ks & 3) ? cx[(ks & 3) - 1][nt] : st[nt], a, bb);
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int c = 8 * nt + 2 * t4;
#pragma unroll
                for (int f = 0; f < 4; ++f) st[nt][f] += (cx[0][nt][f] + cx[1][nt][f]) + cx[2][nt][f];
                St[m0 * SP + c] = tf32_round(st[nt][0]);
                St[m0 * SP + c + 1] = tf32_round(st[nt][1]);
                St[(m0 + 8) * SP + c] = tf32_round(st[nt][2]);
                St[(m0 + 8) * SP + c + 1] = tf32_round(st[nt][3]);
            }
        }
        // (C) state copy updated; this stage is free for block b+2; uniform timeout decision
        if (__syncthreads_or(timed_out)) {   // every thread leaves at the same step
            timed_out = b + 1;
            break;
        }
    }

    if (timed_out) {
        // record the timeout, then wait (bounded) for this CTA's copies still in flight before leaving
        if (t == 0) {
            atomicOr(p.err, 1u);
            const int b = timed_out - 1;
            if (!(b == 0 && p.debug_skip_first_copy == 1)) mbar_wait_bounded(&bar[b & 1], (b >> 1) & 1, p.wait_limit);
            if (b + 1 < nb) mbar_wait_bounded(&bar[(b + 1) & 1], ((b + 1) >> 1) & 1, p.wait_limit);
            if constexpr (kSplit) {   // [W; Qe] of block b (if its wait ran out) and of block b + 1
                mbar_wait_bounded(&bar[2], b & 1, p.wait_limit);
                if (b + 1 < nb) mbar_wait_bounded(&bar[2], (b + 1) & 1, p.wait_limit);
            }
        }
        __syncthreads();
        return;
    }
    float *Scap = s.S_cap ? s.S_cap + (int64_t)h * D * D : nullptr;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int c = 8 * nt + 2 * t4;
        if (owner) {
            Sg[(int64_t)m0 * D + c0 + c] = st[nt][0];
            Sg[(int64_t)m0 * D + c0 + c + 1] = st[nt][1];
            Sg[(int64_t)(m0 + 8) * D + c0 + c] = st[nt][2];
            Sg[(int64_t)(m0 + 8) * D + c0 + c + 1] = st[nt][3];
            if (Scap) {   // the checkpoint of this call's final state
                Scap[(int64_t)m0 * D + c0 + c] = st[nt][0];
                Scap[(int64_t)m0 * D + c0 + c + 1] = st[nt][1];
                Scap[(int64_t)(m0 + 8) * D + c0 + c] = st[nt][2];
                Scap[(int64_t)(m0 + 8) * D + c0 + c + 1] = st[nt][3];
            }
        }
    }
}

template <int D, int DS>
static cudaError_t launch(const LaunchCommon &p, int64_t ch, cudaStream_t st) {
    constexpr size_t smem = ChainPlan<D, DS>::bytes();
    static_assert(smem <= 227 * 1024, "shared memory");
    auto k = chain_tc_kernel<D, DS>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<p.n_sess * p.Hv * (D / DS), kThreads, smem, st>>>(p, ch);
    return cudaGetLastError();
}

template <int D>
static cudaError_t launch_d(const LaunchCommon &p, int64_t ch, cudaStream_t st) {
    // 16 columns per CTA while the launch fits one wave (one CTA per SM): the shortest step for a few
    // chains; 32 columns once it would not, where throughput counts. The arithmetic of every state
    // element is the same in both (same MMAs, same accumulation order), so results do not depend on it.
    static int sms = 0;
    if (!sms) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            sms = 1;
    }
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

cudaError_t gdn_take_device_error(unsigned int *out, cudaStream_t st) {
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(out, g_gdn_device_error, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_gdn_device_error, &zero, sizeof(unsigned int));
}
