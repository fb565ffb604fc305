// The sequential state pass and outputs on the 5th-generation tensor core (tcgen05, accumulators in TMEM),
// bf16-input path, d_k = d_v = 128, over the prologue's fp16 records.
//
// One CTA per chain, i.e. (session, v-head, slice of N columns of d_v), 8 warps. Warp w reads TMEM lanes
// 32 (w % 4) .. 32 (w % 4) + 31 and columns (w / 4) N/2 .. (w / 4) N/2 + N/2 - 1 of each N-column
// accumulator. Per 64-token block, strictly in position order:
//   Z = [W; Qe] S^T              128 x N: one thread issues 8 MMAs (K = 16 each) into TMEM columns [0, N)
//   U' = U - Z[0:64]             lanes 0..63 (warps 0, 1, 4, 5), rounded to fp16 into the B operand of dS
//   O = Z[64:128] + O_intra      lanes 64..127 (warps 2, 3, 6, 7): the output rows, off the dependent path
//   dS = K_tilde^T U'            128 x N: 4 MMAs into TMEM columns [N, 2N), issued once the U' warps are done
//   S^T <- e^{gamma_63} S^T + dS every warp, on the fp32 state rows it holds in registers (TMEM lane = d_k
//                                row), written back as fp16 into the B operand of the next block's Z
// The state enters a block's outputs and its delta-rule correction through W and Qe, and leaves it through
// K_tilde^T U' (the chunked WY form of the recurrence). The fp32 state stays in registers for the whole
// call; shared memory holds only its fp16 copy. Operands are fp16 (the record as the prologue wrote it, U'
// and the state copy rounded here), accumulation fp32. Every element's arithmetic is the same whatever N,
// so the column width per CTA is a launch choice that leaves results unchanged.
//
// A block's record part (48 KB of A operands, then this chain's U and O_intra columns and e^{gamma_63})
// arrives by bulk (TMA) copies into one of two stages, completed on an mbarrier while the block before
// computes. Every mbarrier wait is bounded: on a timeout the CTA records it in the device error word,
// waits (bounded) for its copies and MMAs in flight, frees its TMEM and returns. The CTA also commits its
// share of the session's conv state.
#include "common.cuh"
#include "mma.cuh"
#include "umma.cuh"

namespace gdn {

constexpr int kUChainThreads = 256;
constexpr int kCopier = 64;   // lane 0 of warp 2 (output rows): issues the record copies of blocks 1, 2, ...

template <int N>
struct UChainPlan {
    static_assert(N == 32 || N == 64 || N == 128, "columns per chain");
    static constexpr int NC = N / 2;                         // columns per thread
    static constexpr uint32_t kOps = rec16::kU;              // [W; Qe] and K_tilde^T: the record's first 48 KB
    static constexpr uint32_t kUO = (uint32_t)N * 128;       // the chain's U (or O_intra) columns: N / 8 chunks of 1 KB
    static constexpr uint32_t kEgOff = kOps + 2 * kUO;       // e^{gamma_63} in a stage
    static constexpr uint32_t kTx = kEgOff + 16;             // bytes a stage receives per block
    static constexpr uint32_t kStage = (kTx + 1023) / 1024 * 1024;
    static constexpr uint32_t kSB = 2 * kStage;              // fp16 S^T: B operand of Z, K = 128 (d_k) x N, MN-major
    static constexpr uint32_t kSBO_S = 2048;                 //   LBO 128 (along K), SBO 16 x 128 (along N)
    static constexpr uint32_t kUB = kSB + 128 * N * 2;       // fp16 U': B operand of dS, K = 64 (tokens) x N, MN-major
    static constexpr uint32_t kSBO_U = 1024;                 //   LBO 128, SBO 8 x 128
    static constexpr uint32_t kBar = kUB + 64 * N * 2;       // mbarriers: [0, 1] stages, [2] Z done, [3] dS done
    static constexpr uint32_t kSlot = kBar + 4 * 8;          // TMEM allocation result
    static constexpr uint32_t kBytes = kSlot + 16;
    static constexpr uint32_t kTmemCols = 2 * N < 32 ? 32 : 2 * N;   // Z in [0, N), dS in [N, 2N)
    static_assert(kBytes <= 227 * 1024, "shared memory");
};

// named barrier `id` over n threads (whole warps)
__device__ __forceinline__ void uchain_bar(int id, int n) { asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory"); }

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

template <int N>
__global__ void __launch_bounds__(kUChainThreads, 1) chain_umma_kernel(const __grid_constant__ LaunchCommon p, int64_t ch) {
    using P = UChainPlan<N>;
    constexpr int D = 128, NC = P::NC, nsl = D / N;
    extern __shared__ __align__(1024) unsigned char sm[];
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + P::kBar);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + P::kSlot);
    unsigned char *SB = sm + P::kSB, *UB = sm + P::kUB;

    const int cidx = blockIdx.x;
    const int sl = cidx % nsl, h = (cidx / nsl) % p.Hv;
    const SessRef s = p.s[p.order[cidx / (nsl * p.Hv)]];
    const int c0 = sl * N;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31, q = warp & 3;
    const int row = 32 * q + lane;   // TMEM lane: the token row of Z (U' rows 0..63, output rows 64..127), the d_k row of dS
    const int cl = (warp >> 2) * NC; // this thread's first column within the chain's N
    const int nb = (s.n + kBlock - 1) / kBlock;
    const unsigned char *recs = reinterpret_cast<const unsigned char *>(p.ws_wu);

    grid_dep_launch();   // the next call's prologue may take SMs as this kernel's CTAs leave
    if (t == 0) {
        for (int i = 0; i < 4; ++i) mbar_init(&bar[i], 1);
        mbar_init_fence();
    }
    if (warp == 0) {
        tmem_alloc(tslot, P::kTmemCols);
        tmem_relinquish();
    }
    grid_dep_wait();   // the records of this call, the state and the conv state

    // block b's record part -> stage b & 1 (thread 0 for the first block, thread kCopier for the others)
    auto issue = [&](int b) {
        unsigned char *stg = sm + (b & 1) * P::kStage;
        const unsigned char *r = recs + ((int64_t)(s.blk0 + b) * p.Hv + h) * rec16::kBytes;
        uint64_t *br = &bar[b & 1];
        if (b == 0 && p.debug_skip_first_copy == 1) return;   // test hook: leave the barrier pending
        fence_proxy_async();
        mbar_arrive_expect_tx(br, P::kTx);
#pragma unroll
        for (int k = 0; k < 3; ++k) bulk_g2s(stg + k * 16384, r + k * 16384, 16384, br);
        bulk_g2s(stg + P::kOps, r + rec16::kU + c0 * 128, P::kUO, br);
        bulk_g2s(stg + P::kOps + P::kUO, r + rec16::kO + c0 * 128, P::kUO, br);
        bulk_g2s(stg + P::kEgOff, r + rec16::kEg, 16, br);
    };
    if (t == 0 && nb > 0) issue(0);   // the first block's copies go out first; the rest of the setup overlaps them

    // this chain's share of the session's conv-state commit: the raw inputs at its last three processed positions
    if (s.n > 0) {
        const int ncta = p.Hv * nsl, j = h * nsl + sl;
        const int64_t per = (ch + ncta - 1) / ncta, lo = j * per, hi = lo + per < ch ? lo + per : ch;
        const int64_t nq = (int64_t)p.Hk * D, nv = (int64_t)p.Hv * D;
        __nv_bfloat16 *cs = static_cast<__nv_bfloat16 *>(s.conv);
        const __nv_bfloat16 *cs0 = static_cast<const __nv_bfloat16 *>(s.conv0);
        __nv_bfloat16 *cc = static_cast<__nv_bfloat16 *>(s.conv_cap);
        for (int64_t chan = lo + t; chan < hi; chan += kUChainThreads) {
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

    // the state rows (d_k row `row`, this thread's columns) into registers, and their fp16 copy
    float st[NC];
    {
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
        for (int j = 0; j < NC / 8; ++j) {
            *reinterpret_cast<uint4 *>(SB + ((cl >> 3) + j) * P::kSBO_S + (row >> 3) * 128 + (row & 7) * 16) =
                f8_to_h8(st + 8 * j);
        }
    };
    write_S();
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const uint32_t tl = tmem + ((uint32_t)(32 * q) << 16);   // this warp's lane quarter
    constexpr uint32_t IDESC = umma_idesc_f16(128, N, 0, 1);
    const uint64_t dSB = umma_smem_desc(SB, 128, P::kSBO_S), dUB = umma_smem_desc(UB, 128, P::kSBO_U);
    const uint64_t dWQ[2] = {umma_smem_desc(sm + rec16::kWQ, 128, 2048), umma_smem_desc(sm + P::kStage + rec16::kWQ, 128, 2048)};
    const uint64_t dKT[2] = {umma_smem_desc(sm + rec16::kKT, 128, 1024), umma_smem_desc(sm + P::kStage + rec16::kKT, 128, 1024)};

    int timed_out = 0;
    uint32_t pend = 0;   // thread 0: bit 0 a Z commit, bit 1 a dS commit, issued and not yet seen complete
    for (int b = 0; b < nb; ++b) {
        const unsigned char *stg = sm + (b & 1) * P::kStage;
        bool to = !mbar_wait_bounded(&bar[b & 1], (b >> 1) & 1, p.wait_limit);   // every thread reads the stage
        if (t == 0 && !to) {   // Z = [W; Qe] S^T: K = d_k in 8 steps of 16 (256 bytes along K in both operands)
            tc_fence_after();
            const uint64_t a0 = dWQ[b & 1];
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) umma_bf16(tmem, a0 + 16 * ks, dSB + 16 * ks, IDESC, ks > 0);
            umma_commit(&bar[2]);
            pend |= 1u;
        }
        // the next block's copies, from an output-row warp (off the dependent path); the other stage was
        // released at the end of step b - 1
        if (t == kCopier && b + 1 < nb) issue(b + 1);
        if (!mbar_wait_bounded(&bar[2], b & 1, p.wait_limit)) to = true;
        else if (t == 0) pend &= ~1u;
        tc_fence_after();
        float z[NC];
        tmem_ld_cols<NC>(tl + cl, z);
        if (q < 2) {
            // U' = U - Z[0:64] for token row `row`, as fp16 into the MN-major B operand of dS
            const unsigned char *u = stg + P::kOps + row * 16;
#pragma unroll
            for (int j = 0; j < NC / 8; ++j) {
                float uv[8];
                h8_to_f(*reinterpret_cast<const uint4 *>(u + ((cl >> 3) + j) * 1024), uv);
                const uint4 v = make_uint4(f2_to_h2(uv[0] - z[8 * j], uv[1] - z[8 * j + 1]),
                                           f2_to_h2(uv[2] - z[8 * j + 2], uv[3] - z[8 * j + 3]),
                                           f2_to_h2(uv[4] - z[8 * j + 4], uv[5] - z[8 * j + 5]),
                                           f2_to_h2(uv[6] - z[8 * j + 6], uv[7] - z[8 * j + 7]));
                *reinterpret_cast<uint4 *>(UB + ((cl >> 3) + j) * P::kSBO_U + (row >> 3) * 128 + (row & 7) * 16) = v;
            }
            fence_proxy_async();
            uchain_bar(1, 128);   // warps 0, 1, 4, 5: U' complete
            if (t == 0 && !to) {  // dS = K_tilde^T U': K = 64 tokens in 4 steps
                tc_fence_after();
                const uint64_t a0 = dKT[b & 1];
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) umma_bf16(tmem + N, a0 + 16 * ks, dUB + 16 * ks, IDESC, ks > 0);
                umma_commit(&bar[3]);
                pend |= 2u;
            }
        } else {
            // O = Z[64:128] + O_intra for token row i
            const int i = row - kBlock;
            if (i < s.n - b * kBlock) {
                const unsigned char *oi = stg + P::kOps + P::kUO + i * 16;
                const int64_t o = ((s.row0 + (int64_t)b * kBlock + i) * p.Hv + h) * D + c0 + cl;
#pragma unroll
                for (int j = 0; j < NC / 8; ++j) {
                    float ov[8];
                    h8_to_f(*reinterpret_cast<const uint4 *>(oi + ((cl >> 3) + j) * 1024), ov);
#pragma unroll
                    for (int e = 0; e < 8; ++e) ov[e] += z[8 * j + e];
                    if (p.out_bf16) {
                        const __nv_bfloat162 a = __floats2bfloat162_rn(ov[0], ov[1]), bb = __floats2bfloat162_rn(ov[2], ov[3]),
                                             c = __floats2bfloat162_rn(ov[4], ov[5]), d = __floats2bfloat162_rn(ov[6], ov[7]);
                        *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p.out) + o + 8 * j) =
                            make_uint4(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&bb),
                                       *reinterpret_cast<const uint32_t *>(&c), *reinterpret_cast<const uint32_t *>(&d));
                    } else {
                        float4 *of = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + o + 8 * j);
                        of[0] = make_float4(ov[0], ov[1], ov[2], ov[3]);
                        of[1] = make_float4(ov[4], ov[5], ov[6], ov[7]);
                    }
                }
            }
        }
        if (!mbar_wait_bounded(&bar[3], b & 1, p.wait_limit)) to = true;
        else if (t == 0) pend &= ~2u;
        tc_fence_after();
        {   // S^T <- e^{gamma_63} S^T + dS on this thread's rows, and the fp16 copy for the next block
            float d[NC];
            tmem_ld_cols<NC>(tl + N + cl, d);
            const float e = *reinterpret_cast<const float *>(stg + P::kEgOff);
#pragma unroll
            for (int c = 0; c < NC; ++c) st[c] = fmaf(e, st[c], d[c]);
            write_S();
        }
        fence_proxy_async();
        tc_fence_before();
        // state copy updated, Z and dS read, this stage free for block b + 2; uniform timeout decision
        if (__syncthreads_or(to)) {
            timed_out = b + 1;
            break;
        }
        tc_fence_after();
    }

    if (timed_out) {   // record the timeout, then wait (bounded) for this CTA's copies and MMAs still in flight
        const int b = timed_out - 1;
        if (t == 0) {
            atomicOr(p.err, 1u);
            if (pend & 1u) mbar_wait_bounded(&bar[2], b & 1, p.wait_limit);
            if (pend & 2u) mbar_wait_bounded(&bar[3], b & 1, p.wait_limit);
        }
        if (t == kCopier) {   // block b's copies (unless the test hook held them back) and block b + 1's
            if (!(b == 0 && p.debug_skip_first_copy == 1)) mbar_wait_bounded(&bar[b & 1], (b >> 1) & 1, p.wait_limit);
            if (b + 1 < nb) mbar_wait_bounded(&bar[(b + 1) & 1], ((b + 1) >> 1) & 1, p.wait_limit);
        }
    } else {   // the final state (and its checkpoint)
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

template <int N>
static cudaError_t launch_cols(const LaunchCommon &p, int64_t ch, cudaStream_t st) {
    constexpr size_t smem = UChainPlan<N>::kBytes;
    auto k = chain_umma_kernel<N>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = gdn_launch_pdl(k, p.n_sess * p.Hv * (128 / N), kUChainThreads, smem, st, p, ch);
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
