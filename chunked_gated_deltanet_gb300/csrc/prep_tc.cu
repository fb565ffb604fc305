// Prologue + WY/UT transform on tensor cores (bf16 inputs), one CTA per
// (64-token block, q/k head), for each of the head's G v-heads.
//
// Per block (rows i = 0..63; rows >= n are padding and zero everywhere):
//   conv (kernel 4, halo from the conv state at a call's first block), L2 norm
//   gamma = cumulative log-decay in the block
//   Q K^T, K K^T                                    split-tf32 MMA, lower triangle
//   A_ij = beta_i e^{gamma_i - gamma_j} (K K^T)_ij      (j < i)
//   T = (I + A)^{-1}                                 blocked 16 x 16 inverse, fp32
//   W = T diag(beta e^gamma) K_hat,  U = T diag(beta) V     split-tf32 MMA
//   P_ij = e^{gamma_i - gamma_j} (Q K^T)_ij              (j <= i)
//   Qe = diag(e^gamma) Q_hat - P W,  O_intra = P U          tf32 MMA
//   K_tilde = diag(e^{gamma_63 - gamma_j}) K_hat
// so that, with S0 the state entering the block, the outputs are
// O = Qe S0^T + O_intra and U' = U - W S0^T feeds S^T <- e^{gamma_63} S0^T + K_tilde^T U'.
// The record is written in the fragment order of the state kernel (see common.cuh).
#include "common.cuh"
#include "mma.cuh"

namespace gdn {

template <int D>
__global__ void __launch_bounds__(kThreads, 1) prep_tc_kernel(const LaunchCommon p, int64_t ch) {
    extern __shared__ __align__(16) float smem[];
    constexpr int LQ = D + 4;       // q_hat / k_hat rows: row-indexed A fragments, banks 4g + t
    constexpr int LA = kBlock + 1;  // Q K^T, K K^T
    constexpr int LT = kBlock + 4;  // T, A and P: row-indexed A fragments
    constexpr int LB = D + 8;       // B operands indexed [token][column]: banks 8t + g
    constexpr int RAW = (kBlock + 3) * D;
    float *Yq = smem;
    float *Yk = Yq + kBlock * LQ;
    float *QK = Yk + kBlock * LQ;
    float *KK = QK + kBlock * LA;
    float *Tm = KK + kBlock * LA;
    float *Ps = Tm + kBlock * LT;   // A during the inverse, then P
    float *Bk = Ps + kBlock * LT;   // raw q/k, raw v, inverse scratch, then beta e^gamma k_hat, then W
    float *Bv = Bk + kBlock * LB;   // beta v, then U
    float *gam = Bv + kBlock * LB;
    float *bet = gam + kBlock;
    float *egv = bet + kBlock;
    __nv_bfloat16 *rawq = reinterpret_cast<__nv_bfloat16 *>(Bk);
    __nv_bfloat16 *rawk = rawq + RAW;
    __nv_bfloat16 *rawv = reinterpret_cast<__nv_bfloat16 *>(Bk);
    float *Mt = Bk + (RAW + 1) / 2 + 4;   // inverse scratch, after the raw v tile
    static_assert(2 * RAW * 2 <= kBlock * LB * 4, "q/k raw tiles must fit the Bk region");
    static_assert((RAW + 1) / 2 + 4 + 3 * 16 * 17 <= kBlock * LB, "inverse scratch must fit the Bk region");

    const int blk = blockIdx.x, hk = blockIdx.y, t = threadIdx.x;
    const int warp = t >> 5, lane = t & 31, g8 = lane >> 2, t4 = lane & 3;
    const SessRef s = p.s[find_session(p, blk)];
    const int pos0 = (blk - s.blk0) * kBlock;
    const int n = min(kBlock, s.n - pos0);
    const int64_t row0 = s.row0 + pos0;
    const int Hk = p.Hk, Hv = p.Hv;
    const int64_t nq = (int64_t)Hk * D, nv = (int64_t)Hv * D;
    const __nv_bfloat16 *cw = static_cast<const __nv_bfloat16 *>(p.conv_w);
    const __nv_bfloat16 *cs = static_cast<const __nv_bfloat16 *>(s.conv);

    // Stage rows pos0-3 .. pos0+63 of one head's channels; rows before the call
    // come from the conv state, rows past the block's valid rows are zero.
    auto stage = [&](__nv_bfloat16 *dst, const __nv_bfloat16 *x, int64_t ld, int64_t col0, int64_t chan0) {
        constexpr int CH = D / 8;
        for (int e = t; e < (kBlock + 3) * CH; e += kThreads) {
            const int r = e / CH, c = (e % CH) * 8;
            const int pos = pos0 - 3 + r;
            const void *src;
            int bytes = 16;
            if (pos < 0) src = cs + (int64_t)(3 + pos) * ch + chan0 + c;
            else if (r - 3 < n) src = x + (s.row0 + pos) * ld + col0 + c;
            else { src = x; bytes = 0; }
            cp_async16(dst + r * D + c, src, bytes);
        }
        cp_async_commit();
    };
    auto conv_ch = [&](const __nv_bfloat16 *raw, int c, int64_t chan, float *out, int ldo, const float *rowscale) {
        float w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = __bfloat162float(cw[chan * 4 + i]);
        float h3 = __bfloat162float(raw[c]), h2 = __bfloat162float(raw[D + c]), h1 = __bfloat162float(raw[2 * D + c]);
#pragma unroll 8
        for (int i = 0; i < kBlock; ++i) {
            const float x0 = __bfloat162float(raw[(i + 3) * D + c]);
            const float y = conv_tap<__nv_bfloat16>(w, h3, h2, h1, x0, p.act);
            out[i * ldo + c] = rowscale ? (i < n ? rowscale[i] * y : 0.f) : y;
            h3 = h2; h2 = h1; h1 = x0;
        }
    };

    // 1. q and k: stage, conv, L2 norm
    stage(rawq, static_cast<const __nv_bfloat16 *>(p.xq), nq, (int64_t)hk * D, (int64_t)hk * D);
    stage(rawk, static_cast<const __nv_bfloat16 *>(p.xk), nq, (int64_t)hk * D, nq + (int64_t)hk * D);
    cp_async_wait<0>();
    __syncthreads();
    if (t < 2 * D) {
        const int which = t / D, c = t % D;
        conv_ch(which ? rawk : rawq, c, which * nq + (int64_t)hk * D + c, which ? Yk : Yq, LQ, nullptr);
    }
    __syncthreads();
    for (int r = warp; r < 2 * kBlock; r += kThreads / 32) {
        const int i = r % kBlock;
        float *row = (r < kBlock ? Yq : Yk) + i * LQ;
        float ss = 0.f;
        for (int c = lane; c < D; c += 32) ss = fmaf(row[c], row[c], ss);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float scale = (r < kBlock ? p.q_scale : 1.f) / sqrtf(ss + p.eps);
        for (int c = lane; c < D; c += 32) row[c] = i < n ? row[c] * scale : 0.f;
    }
    __syncthreads();

    // 2. Q K^T and K K^T on the 20 lower-triangle 16x8 tiles, split tf32 (these
    //    dot products of unit vectors can cancel; one rounding would show in short sequences)
    for (int tile = warp; tile < 20; tile += kThreads / 32) {
        int mi = 0, rem = tile;
        while (rem >= 2 * mi + 2) { rem -= 2 * mi + 2; ++mi; }
        const int nj = rem;
        float cq[4] = {0.f, 0.f, 0.f, 0.f}, ck[4] = {0.f, 0.f, 0.f, 0.f};
        const float *qa = Yq + (16 * mi + g8) * LQ + t4;
        const float *ka = Yk + (16 * mi + g8) * LQ + t4;
        const float *kb = Yk + (8 * nj + g8) * LQ + t4;
#pragma unroll 2
        for (int k0 = 0; k0 < D; k0 += 8) {
            uint32_t aqh[4], aql[4], akh[4], akl[4], bh[2], bl[2];
            split_tf32(qa[k0], aqh[0], aql[0]);
            split_tf32(qa[8 * LQ + k0], aqh[1], aql[1]);
            split_tf32(qa[k0 + 4], aqh[2], aql[2]);
            split_tf32(qa[8 * LQ + k0 + 4], aqh[3], aql[3]);
            split_tf32(ka[k0], akh[0], akl[0]);
            split_tf32(ka[8 * LQ + k0], akh[1], akl[1]);
            split_tf32(ka[k0 + 4], akh[2], akl[2]);
            split_tf32(ka[8 * LQ + k0 + 4], akh[3], akl[3]);
            split_tf32(kb[k0], bh[0], bl[0]);
            split_tf32(kb[k0 + 4], bh[1], bl[1]);
            mma_tf32(cq, aql, bh);
            mma_tf32(cq, aqh, bl);
            mma_tf32(cq, aqh, bh);
            mma_tf32(ck, akl, bh);
            mma_tf32(ck, akh, bl);
            mma_tf32(ck, akh, bh);
        }
        const int i0 = 16 * mi + g8, j0 = 8 * nj + 2 * t4;
        QK[i0 * LA + j0] = cq[0]; QK[i0 * LA + j0 + 1] = cq[1];
        QK[(i0 + 8) * LA + j0] = cq[2]; QK[(i0 + 8) * LA + j0 + 1] = cq[3];
        KK[i0 * LA + j0] = ck[0]; KK[i0 * LA + j0 + 1] = ck[1];
        KK[(i0 + 8) * LA + j0] = ck[2]; KK[(i0 + 8) * LA + j0 + 1] = ck[3];
    }

    // 3. each v-head of the group
    for (int gi = 0; gi < p.G; ++gi) {
        const int h = hk * p.G + gi;
        __syncthreads();  // QK/KK written; the previous head's buffers consumed
        stage(rawv, static_cast<const __nv_bfloat16 *>(p.xv), nv, (int64_t)h * D, 2 * nq + (int64_t)h * D);
        if (t < kBlock) {   // gamma: inclusive scan of g (two warps), beta
            float gv = t < n ? p.g[(row0 + t) * Hv + h] : 0.f;
            const float bv = t < n ? p.beta[(row0 + t) * Hv + h] : 0.f;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, gv, o);
                if (lane >= o) gv += y;
            }
            gam[t] = gv;
            bet[t] = bv;
        }
        __syncthreads();
        if (t >= 32 && t < kBlock) gam[t] += gam[31];
        cp_async_wait<0>();
        __syncthreads();
        if (t < kBlock) egv[t] = expf(gam[t]);
        for (int e = t; e < kBlock * kBlock; e += kThreads) {   // A (strict lower) into the P buffer
            const int i = e / kBlock, j = e % kBlock;
            Ps[i * LT + j] = j < i ? bet[i] * expf(gam[i] - gam[j]) * KK[i * LA + j] : 0.f;
        }
        if (t < D) conv_ch(rawv, t, 2 * nq + (int64_t)h * D + t, Bv, LB, bet);   // beta v
        __syncthreads();

        // T = (I + A)^{-1}: diagonal 16x16 blocks by substitution, one column per thread
        if (t < kBlock) {
            const int d = t >> 4, c = t & 15;
            const float *Ad = Ps + 16 * d * LT + 16 * d;
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float sum = 0.f;
#pragma unroll
                for (int j = 0; j < i; ++j)
                    if (j >= c) sum = fmaf(Ad[i * LT + j], x[j], sum);
                x[i] = i < c ? 0.f : (i == c ? 1.f : -sum);
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) Tm[(16 * d + i) * LT + 16 * d + c] = x[i];
        }
        __syncthreads();
        // off-diagonal blocks by distance: T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj
        for (int dist = 1; dist < 4; ++dist) {
            const int nblkd = 4 - dist;
            for (int e = t; e < nblkd * 256; e += kThreads) {
                const int jb = e >> 8, r = (e >> 4) & 15, c = e & 15, ib = jb + dist;
                float sum = 0.f;
                for (int k = 16 * jb; k < 16 * ib; ++k) sum = fmaf(Ps[(16 * ib + r) * LT + k], Tm[k * LT + 16 * jb + c], sum);
                Mt[(jb * 16 + r) * 17 + c] = sum;
            }
            __syncthreads();
            for (int e = t; e < nblkd * 256; e += kThreads) {
                const int jb = e >> 8, r = (e >> 4) & 15, c = e & 15, ib = jb + dist;
                float sum = 0.f;
#pragma unroll
                for (int k = 0; k < 16; ++k) sum = fmaf(Tm[(16 * ib + r) * LT + 16 * ib + k], Mt[(jb * 16 + k) * 17 + c], sum);
                Tm[(16 * ib + r) * LT + 16 * jb + c] = -sum;
            }
            __syncthreads();
        }
        // B operands: beta e^gamma k_hat (over the raw tile and scratch); P over A
        for (int e = t; e < kBlock * D; e += kThreads) {
            const int i = e / D, c = e % D;
            Bk[i * LB + c] = (bet[i] * egv[i]) * Yk[i * LQ + c];
        }
        for (int e = t; e < kBlock * kBlock; e += kThreads) {
            const int i = e / kBlock, j = e % kBlock;
            Ps[i * LT + j] = j <= i ? QK[i * LA + j] * expf(gam[i] - gam[j]) : 0.f;
        }
        __syncthreads();

        float *rec = p.ws_wu + ((int64_t)blk * Hv + h) * rec_floats(D);
        // W = T Bk (warps 0-3) and U = T Bv (warps 4-7), split tf32, T lower triangular
        {
            constexpr int NW = D / 32;   // n-tiles per warp
            const float *B = warp < 4 ? Bk : Bv;
            const int nbase = (warp & 3) * NW * 8;
            float acc[4][NW][4];
#pragma unroll
            for (int mi = 0; mi < 4; ++mi)
#pragma unroll
                for (int nt = 0; nt < NW; ++nt)
#pragma unroll
                    for (int f = 0; f < 4; ++f) acc[mi][nt][f] = 0.f;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint32_t bh[NW][2], bl[NW][2];
#pragma unroll
                for (int nt = 0; nt < NW; ++nt) {
                    const int n0 = nbase + nt * 8 + g8;
                    split_tf32(B[(8 * kk + t4) * LB + n0], bh[nt][0], bl[nt][0]);
                    split_tf32(B[(8 * kk + t4 + 4) * LB + n0], bh[nt][1], bl[nt][1]);
                }
#pragma unroll
                for (int mi = 0; mi < 4; ++mi) {
                    if (mi < kk / 2) continue;
                    const float *ta = Tm + (16 * mi + g8) * LT + 8 * kk + t4;
                    uint32_t ah[4], al[4];
                    split_tf32(ta[0], ah[0], al[0]);
                    split_tf32(ta[8 * LT], ah[1], al[1]);
                    split_tf32(ta[4], ah[2], al[2]);
                    split_tf32(ta[8 * LT + 4], ah[3], al[3]);
#pragma unroll
                    for (int nt = 0; nt < NW; ++nt) {
                        mma_tf32(acc[mi][nt], al, bh[nt]);
                        mma_tf32(acc[mi][nt], ah, bl[nt]);
                        mma_tf32(acc[mi][nt], ah, bh[nt]);
                    }
                }
            }
            __syncthreads();   // every warp is done reading Bk / Bv
            float *dst = warp < 4 ? Bk : Bv;
#pragma unroll
            for (int mi = 0; mi < 4; ++mi)
#pragma unroll
                for (int nt = 0; nt < NW; ++nt) {
                    const int c = nbase + nt * 8 + 2 * t4, i = 16 * mi + g8;
                    dst[i * LB + c] = acc[mi][nt][0];
                    dst[i * LB + c + 1] = acc[mi][nt][1];
                    dst[(i + 8) * LB + c] = acc[mi][nt][2];
                    dst[(i + 8) * LB + c + 1] = acc[mi][nt][3];
                    if (warp >= 4)   // U goes out as-is, in C-fragment slice order
                        *reinterpret_cast<float4 *>(rec + 192 * D + cfrag_slice_index(i, c)) =
                            make_float4(acc[mi][nt][0], acc[mi][nt][1], acc[mi][nt][2], acc[mi][nt][3]);
                }
        }
        __syncthreads();

        // Qe = e^gamma Q_hat - P W and O_intra = P U (tf32): warp w owns n-tiles [w*NT, w*NT + NT) of both
        {
            constexpr int NT = D / 64;
            float aq[4][NT][4], ao[4][NT][4];
#pragma unroll
            for (int mi = 0; mi < 4; ++mi)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int f = 0; f < 4; ++f) aq[mi][nt][f] = ao[mi][nt][f] = 0.f;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint32_t bw[NT][2], bu[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int n0 = (warp * NT + nt) * 8 + g8;
                    bw[nt][0] = tf32_bits(Bk[(8 * kk + t4) * LB + n0]);
                    bw[nt][1] = tf32_bits(Bk[(8 * kk + t4 + 4) * LB + n0]);
                    bu[nt][0] = tf32_bits(Bv[(8 * kk + t4) * LB + n0]);
                    bu[nt][1] = tf32_bits(Bv[(8 * kk + t4 + 4) * LB + n0]);
                }
#pragma unroll
                for (int mi = 0; mi < 4; ++mi) {
                    if (mi < kk / 2) continue;  // P is lower triangular
                    const float *pa = Ps + (16 * mi + g8) * LT + 8 * kk + t4;
                    const uint32_t a[4] = {tf32_bits(pa[0]), tf32_bits(pa[8 * LT]), tf32_bits(pa[4]),
                                           tf32_bits(pa[8 * LT + 4])};
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        mma_tf32(aq[mi][nt], a, bw[nt]);
                        mma_tf32(ao[mi][nt], a, bu[nt]);
                    }
                }
            }
#pragma unroll
            for (int mi = 0; mi < 4; ++mi)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int c = (warp * NT + nt) * 8 + 2 * t4, i = 16 * mi + g8;
                    *reinterpret_cast<float4 *>(rec + 256 * D + cfrag_slice_index(i, c)) =
                        make_float4(ao[mi][nt][0], ao[mi][nt][1], ao[mi][nt][2], ao[mi][nt][3]);
#pragma unroll
                    for (int f = 0; f < 4; ++f) {
                        const int ii = i + 8 * (f >> 1), cc = c + (f & 1);
                        rec[afrag_index(kBlock + ii, cc, D)] = tf32_round(egv[ii] * Yq[ii * LQ + cc] - aq[mi][nt][f]);
                    }
                }
        }
        // W (rows 0..63 of [W; Qe]) and K_tilde^T as A fragments, tf32; e^{gamma_63}
        {
            const float gl = gam[kBlock - 1];
            constexpr int NW4 = 4 * (D / 8) * 32;   // float4 groups of W
            for (int e = t; e < NW4 + (D / 16) * 8 * 32; e += kThreads) {
                const bool isw = e < NW4;
                const int q = isw ? e : e - NW4, ln = q & 31, tile = q >> 5;
                const int gg = ln >> 2, tt = ln & 3;
                float v[4];
                if (isw) {
                    const int mt = tile / (D / 8), ks = tile % (D / 8);
#pragma unroll
                    for (int f = 0; f < 4; ++f)
                        v[f] = tf32_round(Bk[(16 * mt + gg + 8 * (f & 1)) * LB + 8 * ks + tt + 4 * (f >> 1)]);
                    *reinterpret_cast<float4 *>(rec + q * 4) = make_float4(v[0], v[1], v[2], v[3]);
                } else {
                    const int mt = tile >> 3, ks = tile & 7;
#pragma unroll
                    for (int f = 0; f < 4; ++f) {
                        const int m = 16 * mt + gg + 8 * (f & 1), k = 8 * ks + tt + 4 * (f >> 1);
                        v[f] = tf32_round(expf(gl - gam[k]) * Yk[k * LQ + m]);
                    }
                    *reinterpret_cast<float4 *>(rec + 128 * D + q * 4) = make_float4(v[0], v[1], v[2], v[3]);
                }
            }
            if (t == 0) rec[320 * D] = expf(gl);
        }
    }
}

template <int D>
static cudaError_t launch(const LaunchCommon &p, int64_t ch, cudaStream_t st) {
    constexpr int LQ = D + 4, LA = kBlock + 1, LT = kBlock + 4, LB = D + 8;
    constexpr size_t smem =
        sizeof(float) * (2 * kBlock * LQ + 2 * kBlock * LA + 2 * kBlock * LT + 2 * kBlock * LB + 3 * kBlock);
    auto k = prep_tc_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<dim3(p.nblk, p.Hk), kThreads, smem, st>>>(p, ch);
    return cudaGetLastError();
}

}  // namespace gdn

cudaError_t gdn_launch_prep_tc(const gdn::LaunchCommon &p, int D, int64_t ch, cudaStream_t st) {
    return D == 64 ? gdn::launch<64>(p, ch, st) : gdn::launch<128>(p, ch, st);
}
