// The sequential state pass and outputs on the 5th-generation tensor core (tcgen05, accumulators in TMEM),
// bf16-input path, d_k = d_v = 128, over the prologue's fp16 records, as a device function that a kernel
// runs on one CTA per chain: the standalone state kernel (chain_umma.cu), or the chain CTAs of the one-launch
// prefill (prefill_fused.cu), which start each block as soon as the prologue CTAs have published its record.
//
// A chain is (session, v-head, slice of N columns of d_v). Warps 0-7 do the work: warp w reads TMEM lanes
// 32 (w % 4) .. 32 (w % 4) + 31 and columns (w / 4) N/2 .. (w / 4) N/2 + N/2 - 1 of each N-column
// accumulator (further warps of a larger CTA only commit the conv state). Per 64-token block, strictly in
// position order:
//   Z = [W; Qe] S^T              128 x N, K = d_k: threads 0 and 32 each issue 4 MMAs (K = 16 each), into
//                                two accumulators that the epilogue adds (two issuers halve the issue time)
//   U' = U - Z[0:64]             lanes 0..63 (warps 0, 1, 4, 5), rounded to fp16 into the B operand of dS
//   O = Z[64:128] + O_intra      lanes 64..127 (warps 2, 3, 6, 7): the output rows, off the dependent path
//   dS = K_tilde^T U'            128 x N: 4 MMAs (K_tilde^T read MN-major: the record keeps K_tilde by token
//                                rows), issued once the U' warps are done
//   S^T <- e^{gamma_63} S^T + dS warps 0-7, on the fp32 state rows they hold in registers (TMEM lane = d_k
//                                row), written back as fp16 into the B operand of the next block's Z
// The state enters a block's outputs and its delta-rule correction through W and Qe, and leaves it through
// K_tilde^T U' (the chunked WY form of the recurrence). The fp32 state stays in registers for the whole
// call; shared memory holds only its fp16 copy. Operands are fp16 (the record as the prologue wrote it, U'
// and the state copy rounded here), accumulation fp32. Every element's arithmetic is the same whatever N,
// so the column width per CTA is a launch choice that leaves results unchanged.
//
// A block's record part (48 KB of A operands, then this chain's U and O_intra columns and e^{gamma_63})
// arrives by bulk (TMA) copies into one of two stages, completed on an mbarrier while the block before
// computes. Every wait is bounded: on a timeout the CTA records it in the device error word, waits
// (bounded) for its copies and MMAs in flight, frees its TMEM and returns. The CTA also commits the conv
// state of its share of the channels (its q/k head's q and k channels, its v-head's v channels).
#pragma once
#include "common.cuh"
#include "mma.cuh"
#include "umma.cuh"

namespace gdn {

template <int N, int NW = 8>
struct UChainPlan {
    static_assert(N == 32 || N == 64 || N == 128, "columns per chain");
    static_assert(NW == 8 || NW == 16, "worker warps");
    static constexpr int NC = N / (NW / 4);                  // columns per worker thread
    static constexpr uint32_t kOps = rec16::kU;              // [W; Qe] and K_tilde^T: the record's first 48 KB
    static constexpr uint32_t kUO = (uint32_t)N * 128;       // the chain's U (or O_intra) columns: N / 8 chunks of 1 KB
    static constexpr uint32_t kEgOff = kOps + 2 * kUO;       // e^{gamma_63} in a stage
    static constexpr uint32_t kTx = kEgOff + 16;             // bytes a stage receives per block
    static constexpr uint32_t kStage = (kTx + 1023) / 1024 * 1024;
    static constexpr int kS = 2;                             // record stages: the copies run kS - 1 blocks ahead
    static constexpr uint32_t kSB = kS * kStage;             // fp16 S^T: B operand of Z, K = 128 (d_k) x N, MN-major
    static constexpr uint32_t kSBO_S = 2048;                 //   LBO 128 (along K), SBO 16 x 128 (along N)
    static constexpr uint32_t kUB = kSB + 128 * N * 2;       // fp16 U': B operand of dS, K = 64 (tokens) x N, MN-major
    static constexpr uint32_t kSBO_U = 1024;                 //   LBO 128, SBO 8 x 128
    static constexpr uint32_t kBar = kUB + 64 * N * 2;       // mbarriers, indices below
    static constexpr int kFull = 0, kZa = kS, kDS = kS + 1, kZb = kS + 2, kRel = kS + 3, kNBar = 2 * kS + 3;
    // [kFull + i] stage i's copies landed, [kZa] / [kZb] the two halves of Z, [kDS] dS, [kRel + i] stage i released
    static constexpr uint32_t kSlot = kBar + kNBar * 8;      // TMEM allocation result
    static constexpr uint32_t kBytes = kSlot + 16;
    static constexpr uint32_t kTmemCols = N == 32 ? 128 : (N == 64 ? 256 : 512);   // Z halves [0, 2N), dS [2N, 3N)
    static_assert(kBytes <= 227 * 1024, "shared memory");
};

constexpr int kChainWorkThreads = 256;   // the standalone state kernel's CTA: 8 worker warps
// The thread that issues the record copies, kS - 1 blocks ahead (kS record stages). When every warp of the CTA
// is a worker: lane 0 of warp 2 (output rows), inside the step. With spare warps: lane 0 of warp 8, a warp of
// its own that polls the records' publication, paced by the stage-released barriers.
constexpr int kCopier = 64;
constexpr int kOwnCopier = kChainWorkThreads;

// 8 fp32 values in one 32-byte store (dst 32-byte aligned): a whole sector per thread
__device__ __forceinline__ void st_global_v8(float *dst, const float (&v)[8]) {
    asm volatile("st.global.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n" ::"l"(dst), "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]),
                 "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
                 : "memory");
}

// named barrier `id` over n threads (whole warps)
__device__ __forceinline__ void uchain_bar(int id, int n) { asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory"); }
// the same with an OR over the participants' predicates
__device__ __forceinline__ bool uchain_bar_or(int id, int n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n barrier.cta.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// NC consecutive fp32 TMEM columns of this warp's lanes, from column address `ta`
template <int NC>
__device__ __forceinline__ void tmem_ld_cols(uint32_t ta, float (&v)[NC]) {
    uint32_t r[NC / 16][16];
#pragma unroll
    for (int j = 0; j < NC / 16; ++j) tmem_ld16_nowait(ta + 16 * j, r[j]);
#pragma unroll
    for (int j = 0; j < NC / 16; ++j) {
        tmem_wait_ld(r[j]);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[16 * j + i] = __uint_as_float(r[j][i]);
    }
}

// A block's record is always there: the standalone state kernel runs after the prologue kernel.
struct RecordsWritten {
    __device__ __forceinline__ bool operator()(int, int) const { return true; }
};

// The conv-state commit of chain `cidx`'s share of the channels: the q and k channels of its q/k head are split
// over the head group's G x nsl chains, the v channels of its v-head over its nsl slices. Each channel gets the
// raw inputs at the session's last three processed positions. Threads [t0, t0 + nt) of the CTA take part.
template <int N>
__device__ __forceinline__ void chain_conv_commit(const LaunchCommon &p, int64_t ch, const SessRef &s, int h, int sl, int t0,
                                                  int nt) {
    constexpr int D = 128, nsl = D / N;
    const int t = (int)threadIdx.x - t0;
    if (t < 0 || t >= nt || s.n <= 0) return;
    const int hk = h / p.G, gi = h % p.G;
    const int64_t nq = (int64_t)p.Hk * D, nv = (int64_t)p.Hv * D;
    const int parts = p.G * nsl, part = gi * nsl + sl;
    const int qk_per = (2 * D + parts - 1) / parts, v_per = D / nsl;
    __nv_bfloat16 *cs = static_cast<__nv_bfloat16 *>(s.conv);
    const __nv_bfloat16 *cs0 = static_cast<const __nv_bfloat16 *>(s.conv0);
    __nv_bfloat16 *cc = static_cast<__nv_bfloat16 *>(s.conv_cap);
    for (int e = t; e < qk_per + v_per; e += nt) {
        int64_t chan;
        if (e < qk_per) {
            const int i = part * qk_per + e;   // of the head's 2 D q/k channels
            if (i >= 2 * D) continue;
            chan = i < D ? (int64_t)hk * D + i : nq + (int64_t)hk * D + (i - D);
        } else {
            chan = 2 * nq + (int64_t)h * D + sl * v_per + (e - qk_per);
        }
        const __nv_bfloat16 *x;
        int64_t col, ld;
        if (chan < nq) { x = static_cast<const __nv_bfloat16 *>(p.xq); col = chan; ld = nq; }
        else if (chan < 2 * nq) { x = static_cast<const __nv_bfloat16 *>(p.xk); col = chan - nq; ld = nq; }
        else { x = static_cast<const __nv_bfloat16 *>(p.xv); col = chan - 2 * nq; ld = nv; }
        const __nv_bfloat16 o0 = cs0[chan], o1 = cs0[ch + chan], o2 = cs0[2 * ch + chan];
        __nv_bfloat16 nw[3];
#pragma unroll
        for (int r = 0; r < 3; ++r) {
            const int pos = s.n - 3 + r;
            nw[r] = pos >= 0 ? x[(s.row0 + pos) * ld + col] : (pos == -3 ? o0 : (pos == -2 ? o1 : o2));
        }
#pragma unroll
        for (int r = 0; r < 3; ++r) cs[r * ch + chan] = nw[r];
        if (cc) {
#pragma unroll
            for (int r = 0; r < 3; ++r) cc[r * ch + chan] = nw[r];
        }
    }
}

// Chain `cidx` (= ((rank * Hv) + v-head) * (128 / N) + slice, session p.order[rank]) on the CTA's shared memory
// `sm` (UChainPlan<N, NW>::kBytes bytes), with NW worker warps (8 or 16: warp w takes TMEM lane quarter w % 4 and
// column group w / 4). Every thread of the CTA calls it (NT threads, NW * 32 or more). ready(blk, hk)
// is called by the thread that issues the copies of launch block blk (q/k head hk) before it issues them; false
// means it gave up waiting.
// The dependent-launch wait is the caller's.
template <int N, int NT, int NW, class Ready>
__device__ __forceinline__ void chain_run(const LaunchCommon &p, int64_t ch, unsigned char *sm, int cidx, Ready &ready) {
    constexpr int kWT = NW * 32;              // worker threads
    static_assert(NT == kWT || (NW == 8 && NT >= kWT + 64), "threads");
    constexpr bool kOwn = NT > kWT;           // a copier warp of its own, and conv-commit warps
    using P = UChainPlan<N, NW>;
    constexpr int D = 128, NC = P::NC, nsl = D / N;
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + P::kBar);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + P::kSlot);
    unsigned char *SB = sm + P::kSB, *UB = sm + P::kUB;

    const int sl = cidx % nsl, h = (cidx / nsl) % p.Hv;
    const SessRef s = p.s[p.order[cidx / (nsl * p.Hv)]];
    const int c0 = sl * N;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31, q = warp & 3;
    const bool worker = t < kWT;
    const int row = 32 * q + lane;   // TMEM lane: the token row of Z (U' rows 0..63, output rows 64..127), the d_k row of dS
    const int cl = ((warp >> 2) & (NW / 4 - 1)) * NC;   // this thread's first column within the chain's N
    const int nb = (s.n + kBlock - 1) / kBlock;
    const unsigned char *recs = reinterpret_cast<const unsigned char *>(p.ws_wu);

    constexpr int kS = P::kS;
    const int copier = kOwn ? kOwnCopier : kCopier;
    if (t == 0) {
        for (int i = 0; i < P::kNBar; ++i) mbar_init(&bar[i], 1);
        mbar_init_fence();
    }
    if (warp == 0) {
        tmem_alloc(tslot, P::kTmemCols);
        tmem_relinquish();
    }
    __syncthreads();   // barriers initialised (the first copies complete on them)

    // block b's record part -> stage b % kS; false if the record never came
    auto issue = [&](int b) {
        if (!ready(s.blk0 + b, h / p.G)) return false;
        unsigned char *stg = sm + (b % kS) * P::kStage;
        const unsigned char *r = recs + ((int64_t)(s.blk0 + b) * p.Hv + h) * rec16::kBytes;
        uint64_t *br = &bar[P::kFull + b % kS];
        if (b == 0 && p.debug_skip_first_copy == 1) return true;   // test hook: leave the barrier pending
        fence_proxy_async();
        mbar_arrive_expect_tx(br, P::kTx);
#pragma unroll
        for (int k = 0; k < 3; ++k) bulk_g2s(stg + k * 16384, r + k * 16384, 16384, br);
        bulk_g2s(stg + P::kOps, r + rec16::kU + c0 * 128, P::kUO, br);
        bulk_g2s(stg + P::kOps + P::kUO, r + rec16::kO + c0 * 128, P::kUO, br);
        bulk_g2s(stg + P::kEgOff, r + rec16::kEg, 16, br);
        return true;
    };
    __shared__ int s_ready0;   // block 0's record (and with it the session's first-block halo reads) is done
    int issued = -1;           // the copier: the last block whose copies it issued
    if (t == copier) {         // the first kS - 1 blocks (a larger CTA's copier carries on in its own loop)
        bool ok = true;
        for (int b = 0; b < nb && b < (kOwn ? 1 : kS - 1) && ok; ++b)
            if ((ok = issue(b))) issued = b;
        s_ready0 = nb > 0 ? (int)(issued >= 0) : 1;
    }

    // the state rows (d_k row `row`, this thread's columns) into registers, and their fp16 copy
    float st[NC];
    if (worker) {
        const float *Sg0 = s.S0 + ((int64_t)h * D + row) * D + c0 + cl;
#pragma unroll
        for (int c = 0; c < NC; c += 4) {
            const float4 v = *reinterpret_cast<const float4 *>(Sg0 + c);
            st[c] = v.x; st[c + 1] = v.y; st[c + 2] = v.z; st[c + 3] = v.w;
        }
    }
    // MN-major B operand of Z: the 8 columns n..n+7 of d_k row k form one 16-byte row of a core matrix
    auto write_S = [&]() {
#pragma unroll
        for (int j = 0; j < NC / 8; ++j)
            *reinterpret_cast<uint4 *>(SB + ((cl >> 3) + j) * P::kSBO_S + (row >> 3) * 128 + (row & 7) * 16) =
                f8_to_h8(st + 8 * j);
    };
    if (worker) write_S();
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    int timed_out = s_ready0 ? 0 : 1;
    if (timed_out && t == 0) atomicOr(p.err, 1u);
    // the conv state (the first block's record is published, so every halo read of the session's first block is
    // done): by the warps after the copier's beside the block loop; with 8 workers and no spare warps by every
    // thread before the loop; with 16 workers after it
    if constexpr (kOwn) {
        if (warp > kOwnCopier / 32 && !timed_out) chain_conv_commit<N>(p, ch, s, h, sl, kOwnCopier + 32, NT - kOwnCopier - 32);
    } else if constexpr (NW == 8) {
        if (!timed_out) chain_conv_commit<N>(p, ch, s, h, sl, 0, NT);
    }
    // the copier warp: blocks 1, 2, ... in order, each once its stage is released (block b - kS done) and its
    // record published; afterwards it waits (bounded) until its last copies have landed
    if constexpr (kOwn) {
        if (t == kOwnCopier && !timed_out) {
            bool ok = true;
            for (int b = 1; b < nb && ok; ++b) {
                if (b >= kS && !mbar_wait_bounded(&bar[P::kRel + b % kS], ((b - kS) / kS) & 1, p.wait_limit)) ok = false;
                if (ok && !issue(b)) ok = false;
                if (ok) issued = b;
            }
            if (!ok) atomicOr(p.err, 1u);   // the block loop's waits then run out as well
            for (int b = issued - kS + 1 > 0 ? issued - kS + 1 : 0; b <= issued; ++b)
                if (!(b == 0 && p.debug_skip_first_copy == 1))
                    mbar_wait_bounded(&bar[P::kFull + b % kS], (b / kS) & 1, p.wait_limit);
        }
    }
    const uint32_t tmem = *tslot;
    const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);   // this warp's lane quarter
    constexpr uint32_t IDESC = umma_idesc_f16(128, N, 0, 1);      // Z: A K-major, B MN-major
    constexpr uint32_t IDESC_DS = umma_idesc_f16(128, N, 1, 1);   // dS: both MN-major
    const uint64_t dSB = umma_smem_desc(SB, 128, P::kSBO_S), dUB = umma_smem_desc(UB, 128, P::kSBO_U);
    // the stages' A operands: stage i's descriptors are stage 0's plus i stage sizes (in 16-byte units)
    const uint64_t dWQ0 = umma_smem_desc(sm + rec16::kWQ, 128, 2048), dKT0 = umma_smem_desc(sm + rec16::kKT, 2048, 128);
    constexpr uint64_t kStageDesc = P::kStage >> 4;

    uint32_t pend = 0;   // threads 0 and 32: bit 0 a Z commit, bit 1 a dS commit, issued and not yet seen complete
    bool copy_next = false;   // kCopier: the copies of block b + kS - 1 went out
    if (worker && !timed_out) {
        for (int b = 0; b < nb; ++b) {
            const int si = b % kS;
            const unsigned char *stg = sm + si * P::kStage;
            bool to = !mbar_wait_bounded(&bar[P::kFull + si], (b / kS) & 1, p.wait_limit);   // every worker reads the stage
            if ((t == 0 || t == 32) && !to) {   // Z = [W; Qe] S^T, K = d_k: 4 steps of 16 per issuer (256 bytes each)
                tc_fence_after();
                const int k0 = t == 0 ? 0 : 4;
                const uint64_t a0 = dWQ0 + si * kStageDesc + 16 * k0, b0 = dSB + 16 * k0;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) umma_bf16(tmem + (t == 0 ? 0 : N), a0 + 16 * ks, b0 + 16 * ks, IDESC, ks > 0);
                umma_commit(&bar[t == 0 ? P::kZa : P::kZb]);
                pend |= 1u;
            }
            // block b + kS - 1's copies, from an output-row warp (off the dependent path); its stage was released
            // at the end of step b - 1
            if (!kOwn && t == kCopier) {
                copy_next = b + kS - 1 >= nb || issue(b + kS - 1);
                if (copy_next && b + kS - 1 < nb) issued = b + kS - 1;
            }
            {
                const bool za = mbar_wait_bounded(&bar[P::kZa], b & 1, p.wait_limit);
                const bool zb = mbar_wait_bounded(&bar[P::kZb], b & 1, p.wait_limit);
                if (!za || !zb) to = true;
                if ((t == 0 && za) || (t == 32 && zb)) pend &= ~1u;
            }
            tc_fence_after();
            // Z in 16-column chunks (the two halves added): U' rows -> the B operand of dS, output rows -> out
            const int i = row - kBlock;
            const unsigned char *uo = stg + P::kOps + (q < 2 ? 0u : P::kUO) + (q < 2 ? row : i) * 16;
            const bool out_row = q >= 2 && i < s.n - b * kBlock;
            const int64_t o = ((s.row0 + (int64_t)b * kBlock + i) * p.Hv + h) * D + c0 + cl;
            // 32-byte stores where the output allows them (every 8-column group of a row starts on a 32-byte
            // boundary when the output does)
            const bool out32 = (reinterpret_cast<uintptr_t>(p.out) & 31) == 0;
            // with up to 32 columns per thread every TMEM load of the step goes out before the one wait
            constexpr bool kAllAtOnce = NC <= 32;
            float zall[kAllAtOnce ? NC : 1];
            if constexpr (kAllAtOnce) {
                uint32_t ra[NC / 16][16], rb[NC / 16][16];
#pragma unroll
                for (int j16 = 0; j16 < NC / 16; ++j16) {
                    tmem_ld16_nowait(tl + cl + 16 * j16, ra[j16]);
                    tmem_ld16_nowait(tl + N + cl + 16 * j16, rb[j16]);
                }
#pragma unroll
                for (int j16 = 0; j16 < NC / 16; ++j16) {
                    tmem_wait_ld(ra[j16]);
                    tmem_wait_ld(rb[j16]);
#pragma unroll
                    for (int c = 0; c < 16; c += 2)   // packed pairs: each lane rounds as the scalar add does
                        f2_unpack(f2_add(f2_pack(__uint_as_float(ra[j16][c]), __uint_as_float(ra[j16][c + 1])),
                                         f2_pack(__uint_as_float(rb[j16][c]), __uint_as_float(rb[j16][c + 1]))),
                                  zall[16 * j16 + c], zall[16 * j16 + c + 1]);
                }
            }
#pragma unroll
            for (int j16 = 0; j16 < NC / 16; ++j16) {
                float z[16];
                if constexpr (kAllAtOnce) {
#pragma unroll
                    for (int c = 0; c < 16; ++c) z[c] = zall[16 * j16 + c];
                } else {
                    uint32_t ra[16], rb[16];
                    tmem_ld16_nowait(tl + cl + 16 * j16, ra);
                    tmem_ld16_nowait(tl + N + cl + 16 * j16, rb);
                    tmem_wait_ld(ra);
                    tmem_wait_ld(rb);
#pragma unroll
                    for (int c = 0; c < 16; ++c) z[c] = __uint_as_float(ra[c]) + __uint_as_float(rb[c]);
                }
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int j = 2 * j16 + hf;   // 8-column chunk of this thread's columns
                    float v[8];
                    h8_to_f(*reinterpret_cast<const uint4 *>(uo + ((cl >> 3) + j) * 1024), v);
                    if (q < 2) {   // U' = U - Z[0:64] for token row `row`, as fp16 into the MN-major B operand of dS
#pragma unroll
                        for (int e = 0; e < 8; e += 2)   // v - z as one rounding: fma(z, -1, v)
                            f2_unpack(f2_fma(f2_pack(z[8 * hf + e], z[8 * hf + e + 1]), f2_pack(-1.f, -1.f), f2_pack(v[e], v[e + 1])),
                                      v[e], v[e + 1]);
                        *reinterpret_cast<uint4 *>(UB + ((cl >> 3) + j) * P::kSBO_U + (row >> 3) * 128 + (row & 7) * 16) =
                            f8_to_h8(v);
                    } else if (out_row) {   // O = Z[64:128] + O_intra for token row i
#pragma unroll
                        for (int e = 0; e < 8; e += 2)
                            f2_unpack(f2_add(f2_pack(v[e], v[e + 1]), f2_pack(z[8 * hf + e], z[8 * hf + e + 1])), v[e], v[e + 1]);
                        if (p.out_bf16) {
                            const __nv_bfloat162 a = __floats2bfloat162_rn(v[0], v[1]), bb = __floats2bfloat162_rn(v[2], v[3]),
                                                 c = __floats2bfloat162_rn(v[4], v[5]), d = __floats2bfloat162_rn(v[6], v[7]);
                            *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.out) + o + 8 * j) =
                                make_uint4(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&bb),
                                           *reinterpret_cast<const uint32_t *>(&c), *reinterpret_cast<const uint32_t *>(&d));
                        } else if (out32) {
                            st_global_v8(static_cast<float *>(p.out) + o + 8 * j, v);
                        } else {
                            float4 *of = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + o + 8 * j);
                            of[0] = make_float4(v[0], v[1], v[2], v[3]);
                            of[1] = make_float4(v[4], v[5], v[6], v[7]);
                        }
                    }
                }
            }
            if (q < 2) {
                fence_proxy_async();
                uchain_bar(1, kWT / 2);   // the U' warps (lane quarters 0 and 1): U' complete
                if (t == 0 && !to) {  // dS = K_tilde^T U': K = 64 tokens in 4 steps
                    tc_fence_after();
                    const uint64_t a0 = dKT0 + si * kStageDesc;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) umma_bf16(tmem + 2 * N, a0 + 256 * ks, dUB + 16 * ks, IDESC_DS, ks > 0);
                    umma_commit(&bar[P::kDS]);
                    pend |= 2u;
                }
            }
            if (!mbar_wait_bounded(&bar[P::kDS], b & 1, p.wait_limit)) to = true;
            else if (t == 0) pend &= ~2u;
            tc_fence_after();
            {   // S^T <- e^{gamma_63} S^T + dS on this thread's rows, and the fp16 copy for the next block
                float d[NC];
                tmem_ld_cols<NC>(tl + 2 * N + cl, d);
                const float e = *reinterpret_cast<const float *>(stg + P::kEgOff);
                const uint64_t e2 = f2_pack(e, e);
#pragma unroll
                for (int c = 0; c < NC; c += 2) f2_unpack(f2_fma(e2, f2_pack(st[c], st[c + 1]), f2_pack(d[c], d[c + 1])), st[c], st[c + 1]);
                write_S();
            }
            fence_proxy_async();
            tc_fence_before();
            // warps 0-7: state copy updated, Z and dS read, this stage free for block b + 2; uniform timeout
            // decision (a copy that was never issued counts as one)
            if (uchain_bar_or(2, kWT, to || (!kOwn && t == kCopier && !copy_next))) {
                timed_out = b + 1;
                break;
            }
            if (kOwn && t == 0) mbar_arrive(&bar[P::kRel + si]);   // stage si released (for block b + kS)
            tc_fence_after();
        }
    }

    if (timed_out && worker) {   // record the timeout, then wait (bounded) for this CTA's copies and MMAs in flight
        const int b = timed_out - 1;
        if (t == 0) atomicOr(p.err, 1u);
        if (t == 0 || t == 32) {
            if (pend & 1u) mbar_wait_bounded(&bar[t == 0 ? P::kZa : P::kZb], b & 1, p.wait_limit);
            if (pend & 2u) mbar_wait_bounded(&bar[P::kDS], b & 1, p.wait_limit);
        }
        if (!kOwn && t == kCopier)   // blocks b .. issued (unless the test hook held block 0 back)
            for (int j = b; j <= issued; ++j)
                if (!(j == 0 && p.debug_skip_first_copy == 1))
                    mbar_wait_bounded(&bar[P::kFull + j % kS], (j / kS) & 1, p.wait_limit);
    } else if (worker) {   // the final state (and its checkpoint)
        if constexpr (!kOwn && NW == 16) chain_conv_commit<N>(p, ch, s, h, sl, 0, kWT);
        float *Sg = s.S + ((int64_t)h * D + row) * D + c0 + cl;
        float *Sc = s.S_cap ? s.S_cap + ((int64_t)h * D + row) * D + c0 + cl : nullptr;
#pragma unroll
        for (int c = 0; c < NC; c += 4) {
            const float4 v = make_float4(st[c], st[c + 1], st[c + 2], st[c + 3]);
            *reinterpret_cast<float4 *>(Sg + c) = v;
            if (Sc) *reinterpret_cast<float4 *>(Sc + c) = v;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, P::kTmemCols);
}

}  // namespace gdn
