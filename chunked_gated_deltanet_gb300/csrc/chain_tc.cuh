// The sequential state pass and outputs on tensor cores (bf16-input path), as
// pieces that a kernel composes: one chain is (session, v-head, slice of DS
// columns of d_v), walking the session's 64-token blocks strictly in position
// order. Per block:
//   Z = [W; Qe] S^T                  (128 x DS; warp w owns rows 16w..16w+15)
//   U' = U - Z[0:64],  O = Z[64:128] + O_intra   (outputs written here)
//   S^T <- e^{gamma_63} S^T + K_tilde^T U'        (warp w owns state rows 16w..16w+15)
// The fp32 state lives in the registers of the warps that own its rows (in
// m16n8 accumulator layout); shared memory holds its tf32 copy, the B operand
// of the next block's first product. Operands are tf32 (rounded by the
// prologue, or here for U'), accumulation is fp32. The prologue stores each
// block's operands in fragment order, so a block is a few contiguous bulk
// copies (TMA) issued by one thread into a two-stage buffer and completed on
// an mbarrier. The compute runs on the CTA's 8 warps (kThreads threads).
#pragma once
#include "common.cuh"
#include "mma.cuh"

namespace gdn {

// Shared-memory plan of a chain with DS state columns. With 16 columns both operand sets of a block (A of
// the first product, [W; Qe], and of the second, K_tilde^T, with the U and O_intra slices) are double
// buffered. With 32 columns that does not fit: the K_tilde^T part stays double buffered and [W; Qe] has
// one buffer, refilled for the next block while the second product runs.
template <int D, int DS>
struct ChainPlan {
    static constexpr bool kSplit = DS > kSliceCols;
    static constexpr int SP = DS + 8;          // tf32 S^T and U' rows (B fragments): banks 8t + g, distinct
    static constexpr int WQF = 2 * kBlock * D; // [W; Qe] fragments
    static constexpr int KTF = kBlock * D;     // K_tilde^T fragments
    static constexpr int UF = kBlock * DS;     // U (or O_intra) fragments of the chain's columns
    static constexpr int KSTAGE = KTF + 2 * UF + 4;                        // K_tilde^T, U, O_intra, e^{gamma_63}
    static constexpr int STAGE = kSplit ? KSTAGE : WQF + KSTAGE;           // one double-buffered stage
    static constexpr int WQBUF = kSplit ? WQF : 0;                         // the single [W; Qe] buffer
    static constexpr size_t bytes() {
        return sizeof(float) * (2 * STAGE + WQBUF + D * SP + kBlock * SP) + 4 * sizeof(uint64_t);
    }
};

// Barrier of the chain's compute warps (all of the CTA's 8 warps).
__device__ __forceinline__ void chain_bar() { asm volatile("bar.sync 1, %0;\n" ::"n"(kThreads) : "memory"); }

template <int D, int DS>
struct Chain {
    using P = ChainPlan<D, DS>;
    static constexpr int NT = DS / 8, SP = P::SP, WQF = P::WQF, KTF = P::KTF, UF = P::UF, STAGE = P::STAGE;
    static constexpr bool kSplit = P::kSplit;
    static constexpr int nsl = D / DS;
    static_assert(D == 128 || D == 64, "head dim");
    static_assert(DS == 16 || DS == 32, "slice width");

    const LaunchCommon &p;
    float *smem, *wqbuf, *St, *Ups;
    uint64_t *bar;   // [0..1] stages, [2] the [W; Qe] buffer (split plan)
    SessRef s;
    int sl, h, c0, t, warp, lane, g8, t4, nb, m0;
    bool owner;      // this warp owns state rows 16w..16w+15
    float st[NT][4]; // the state rows of this thread (accumulator layout)

    // chain index cidx = ((rank * Hv) + v-head) * (D / DS) + slice, session p.order[rank]
    __device__ __forceinline__ Chain(const LaunchCommon &p_, float *smem_, int cidx) : p(p_), smem(smem_) {
        wqbuf = smem + 2 * STAGE;
        St = wqbuf + P::WQBUF;
        Ups = St + D * SP;
        bar = reinterpret_cast<uint64_t *>(Ups + kBlock * SP);
        sl = cidx % nsl;
        h = (cidx / nsl) % p.Hv;
        s = p.s[p.order[cidx / (nsl * p.Hv)]];
        c0 = sl * DS;
        t = threadIdx.x; warp = t >> 5; lane = t & 31; g8 = lane >> 2; t4 = lane & 3;
        nb = (s.n + kBlock - 1) / kBlock;
        owner = 16 * warp < D;
        m0 = 16 * warp + g8;
    }
    // block b's operands: A of the first product, then K_tilde^T, U, O_intra, e^{gamma_63}
    __device__ __forceinline__ const float *wq_of(int b) const { return kSplit ? wqbuf : smem + (b & 1) * STAGE; }
    __device__ __forceinline__ const float *kt_of(int b) const { return smem + (b & 1) * STAGE + (kSplit ? 0 : WQF); }
    __device__ __forceinline__ const float *record(int b) const {
        return p.ws_wu + ((int64_t)(s.blk0 + b) * p.Hv + h) * rec_floats(D);
    }

    // The chain's share of the session's conv-state commit (the raw inputs at the session's last three
    // processed positions); the shares of all chains of the session cover every channel once.
    __device__ __forceinline__ void conv_commit(int64_t ch) const {
        const int ncta = p.Hv * nsl, j = h * nsl + sl;
        const int64_t per = (ch + ncta - 1) / ncta, chan = j * per + t;
        if (t < per && chan < ch && s.n > 0) {
            const int64_t nq = (int64_t)p.Hk * D, nv = (int64_t)p.Hv * D;
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

    // thread 0: block b's operands -> stage b & 1 (with the 16-column plan all of them, with the split plan
    // the K_tilde^T part; [W; Qe] goes through issue_wq)
    static constexpr int CHUNK = 4096;   // floats per bulk copy (16 KB)
    static_assert(WQF % CHUNK == 0 && KTF % CHUNK == 0, "operand blocks are whole numbers of chunks");
    __device__ __forceinline__ void issue(int b) {
        float *buf = smem + (b & 1) * STAGE;
        const float *r = record(b);
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
    }
    __device__ __forceinline__ void issue_wq(int b) {   // split plan: [W; Qe] of block b into its single buffer
        const float *r = record(b);
        fence_proxy_async();
        mbar_arrive_expect_tx(&bar[2], (uint32_t)sizeof(float) * WQF);
#pragma unroll
        for (int q = 0; q < WQF / CHUNK; ++q) bulk_g2s(wqbuf + q * CHUNK, r + q * CHUNK, sizeof(float) * CHUNK, &bar[2]);
    }
    __device__ __forceinline__ void init_bars() {   // thread 0
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        mbar_init(&bar[2], 1);
        mbar_init_fence();
    }

    // the tf32 copy of this thread's state rows into shared memory
    __device__ __forceinline__ void write_St() {
        if (!owner) return;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int c = 8 * nt + 2 * t4;
            St[m0 * SP + c] = tf32_round(st[nt][0]);
            St[m0 * SP + c + 1] = tf32_round(st[nt][1]);
            St[(m0 + 8) * SP + c] = tf32_round(st[nt][2]);
            St[(m0 + 8) * SP + c + 1] = tf32_round(st[nt][3]);
        }
    }
    // the starting state (the session's own, or a prefix's) into registers and its tf32 copy
    __device__ __forceinline__ void load_state() {
        const float *Sg0 = s.S0 + (int64_t)h * D * D;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int c = 8 * nt + 2 * t4;
            if (owner) {
                st[nt][0] = Sg0[(int64_t)m0 * D + c0 + c];
                st[nt][1] = Sg0[(int64_t)m0 * D + c0 + c + 1];
                st[nt][2] = Sg0[(int64_t)(m0 + 8) * D + c0 + c];
                st[nt][3] = Sg0[(int64_t)(m0 + 8) * D + c0 + c + 1];
            } else {
                st[nt][0] = st[nt][1] = st[nt][2] = st[nt][3] = 0.f;
            }
        }
        write_St();
    }

    // Block b on warps 0-7, its operands issued: true if a bounded wait ran out (the step still runs, on
    // whatever the stage holds; the caller acts on a timeout after its end-of-step barrier). With the split
    // plan thread 0 also refills [W; Qe] for block b + 1 once the first product is done.
    __device__ __forceinline__ bool step(int b) {
        bool timed_out = false;
        const float *wq = wq_of(b), *kt = kt_of(b), *uo0 = kt + KTF;
        // every thread acquires the stage itself
        if (!mbar_wait_bounded(&bar[b & 1], (b >> 1) & 1, p.wait_limit)) timed_out = true;
        if constexpr (kSplit)
            if (!mbar_wait_bounded(&bar[2], b & 1, p.wait_limit)) timed_out = true;

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
                        const int64_t oi = ((s.row0 + (int64_t)b * kBlock + ii) * p.Hv + h) * D + c0 + c;
                        if (p.out_bf16)
                            *reinterpret_cast<__nv_bfloat162 *>(static_cast<__nv_bfloat16 *>(p.out) + oi) =
                                __floats2bfloat162_rn(o0, o1);
                        else
                            *reinterpret_cast<float2 *>(static_cast<float *>(p.out) + oi) = make_float2(o0, o1);
                    }
                }
            }
        }
        chain_bar();  // (B) U' complete; every read of the tf32 state copy and of [W; Qe] done
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
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int f = 0; f < 4; ++f) st[nt][f] += (cx[0][nt][f] + cx[1][nt][f]) + cx[2][nt][f];
            write_St();
        }
        return timed_out;
    }

    // thread 0, after a timeout at block b: wait (bounded) for this chain's copies still in flight
    // (those of block b, and of block b + 1 when `next_issued`)
    __device__ __forceinline__ void drain(int b, bool next_issued) {
        if (!(b == 0 && p.debug_skip_first_copy == 1)) mbar_wait_bounded(&bar[b & 1], (b >> 1) & 1, p.wait_limit);
        if (next_issued) mbar_wait_bounded(&bar[(b + 1) & 1], ((b + 1) >> 1) & 1, p.wait_limit);
        if constexpr (kSplit) {   // [W; Qe] of block b (if its wait ran out) and of block b + 1
            mbar_wait_bounded(&bar[2], b & 1, p.wait_limit);
            if (b + 1 < nb) mbar_wait_bounded(&bar[2], (b + 1) & 1, p.wait_limit);
        }
    }

    // the final state (and its checkpoint) from the owner warps' registers
    __device__ __forceinline__ void finish() const {
        if (!owner) return;
        float *Sg = s.S + (int64_t)h * D * D;
        float *Scap = s.S_cap ? s.S_cap + (int64_t)h * D * D : nullptr;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const int c = 8 * nt + 2 * t4;
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
};

}  // namespace gdn
