// Prologue + WY/UT transform on tensor cores (bf16 inputs), one CTA per
// (64-token block, q/k head), for each of the head's G v-heads.
//
// Per block (rows i = 0..63; rows >= n are padding and zero everywhere):
//   conv (kernel 4, halo from the conv state at a call's first block), L2 norm
//   gamma = cumulative log-decay in the block
//   QK^T, KK^T                                     split-tf32 MMA (lower triangle only)
//   A_ij = beta_i e^{gamma_i - gamma_j} (K K^T)_ij      (j < i)
//   P_ij = e^{gamma_i - gamma_j} (Q K^T)_ij             (j <= i)
//   (I + A) [W | U] = [diag(beta e^gamma) K_hat | diag(beta) V]   forward substitution
//   Qe = diag(e^gamma) Q_hat - P W,  O_intra = P U       tf32 MMA
//   K_tilde = diag(e^{gamma_63 - gamma_j}) K_hat
// so that, with S0 the state entering the block, the outputs are
// O = Qe S0^T + O_intra and U' = U - W S0^T feeds S^T <- e^{gamma_63} S0^T + K_tilde^T U'.
// Record per (block, v-head), in floats: [W; Qe] [128][D] and K_tilde [64][D]
// (both pre-rounded to tf32), U [64][D], O_intra [64][D], e^{gamma_63}.
#include "common.cuh"
#include "mma.cuh"

namespace gdn {

template <int D>
__global__ void __launch_bounds__(kThreads, 1) prep_tc_kernel(const LaunchCommon p, int64_t ch) {
    extern __shared__ __align__(16) float smem[];
    constexpr int LQ = D + 4;       // q_hat / k_hat rows: A-fragment reads hit 32 distinct banks
    constexpr int LA = kBlock + 1;  // 64 x 64 tiles written from fragments / read as scalars
    constexpr int LX = 2 * D + 8;   // [W | U]: B-fragment reads hit 32 distinct banks
    constexpr int LP = kBlock + 4;  // P: A-fragment reads
    constexpr int RAW = (kBlock + 3) * D;  // raw bf16 tile, halo rows first
    float *Yq = smem;
    float *Yk = Yq + kBlock * LQ;
    float *QK = Yk + kBlock * LQ;
    float *KK = QK + kBlock * LA;
    float *Am = KK + kBlock * LA;
    float *X = Am + kBlock * LA;
    float *Ps = X + kBlock * LX;
    float *gam = Ps + kBlock * LP;
    float *bet = gam + kBlock;
    float *eg = bet + kBlock;
    // raw input tiles alias regions that are free at the time
    __nv_bfloat16 *rawq = reinterpret_cast<__nv_bfloat16 *>(X);
    __nv_bfloat16 *rawk = rawq + RAW;
    __nv_bfloat16 *rawv = reinterpret_cast<__nv_bfloat16 *>(Ps);
    static_assert(2 * RAW * 2 <= kBlock * LX * 4, "q/k raw tiles must fit the X region");
    static_assert(RAW * 2 <= kBlock * LP * 4, "v raw tile must fit the P region");

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

    // Stage rows pos0-3 .. pos0+63 of one head's channels into shared memory.
    // Rows before the call come from the conv state; rows past the block's valid
    // rows are zero-filled.
    auto stage = [&](__nv_bfloat16 *dst, const __nv_bfloat16 *x, int64_t ld, int64_t col0, int64_t chan0) {
        constexpr int CH = D / 8;  // 16-byte chunks per row
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
    // Conv of channel c of a staged tile into out[i * ldo + c] * scale_i (scale 1 if null).
    auto conv_ch = [&](const __nv_bfloat16 *raw, int c, int64_t chan, float *out, int ldo, const float *rowscale) {
        float w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = __bfloat162float(cw[chan * 4 + i]);
        float h3 = __bfloat162float(raw[0 * D + c]), h2 = __bfloat162float(raw[1 * D + c]);
        float h1 = __bfloat162float(raw[2 * D + c]);
#pragma unroll 8
        for (int i = 0; i < kBlock; ++i) {
            const float x0 = __bfloat162float(raw[(i + 3) * D + c]);
            const float y = conv_tap<__nv_bfloat16>(w, h3, h2, h1, x0, p.act);
            out[i * ldo + c] = rowscale ? (i < n ? rowscale[i] * y : 0.f) : y;
            h3 = h2; h2 = h1; h1 = x0;
        }
    };

    // 1. q and k tiles -> conv
    stage(rawq, static_cast<const __nv_bfloat16 *>(p.xq), nq, (int64_t)hk * D, (int64_t)hk * D);
    stage(rawk, static_cast<const __nv_bfloat16 *>(p.xk), nq, (int64_t)hk * D, nq + (int64_t)hk * D);
    cp_async_wait<0>();
    __syncthreads();
    if (t < 2 * D) {
        const int which = t / D, c = t % D;
        conv_ch(which ? rawk : rawq, c, which * nq + (int64_t)hk * D + c, which ? Yk : Yq, LQ, nullptr);
    }
    __syncthreads();

    // 2. L2 norm per row; padding rows zero
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

    // 3. QK^T and KK^T on the 20 lower-triangle 16x8 tiles (m-tile mi, n-tile nj <= 2 mi + 1)
    for (int tile = warp; tile < 20; tile += kThreads / 32) {
        int mi = 0, rem = tile;
        while (rem >= 2 * mi + 2) { rem -= 2 * mi + 2; ++mi; }
        const int nj = rem;
        float cq[4] = {0.f, 0.f, 0.f, 0.f}, ck[4] = {0.f, 0.f, 0.f, 0.f};
        const float *qa = Yq + (16 * mi + g8) * LQ + t4;
        const float *ka = Yk + (16 * mi + g8) * LQ + t4;
        const float *kb = Yk + (8 * nj + g8) * LQ + t4;
        // split tf32 (hi*hi + hi*lo + lo*hi): these dot products of unit vectors can cancel,
        // and a single rounding of the operands would show in short sequences
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

    // 4. each v-head of the group
    for (int gi = 0; gi < p.G; ++gi) {
        const int h = hk * p.G + gi;
        __syncthreads();  // QK/KK written; the previous head's X and P consumed
        stage(rawv, static_cast<const __nv_bfloat16 *>(p.xv), nv, (int64_t)h * D, 2 * nq + (int64_t)h * D);
        // gamma: inclusive scan of g over the block (two warps), beta
        if (t < kBlock) {
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
        if (t < kBlock) eg[t] = expf(gam[t]);
        // A (strict lower), rhs of W, v conv -> rhs of U
        for (int e = t; e < kBlock * kBlock; e += kThreads) {
            const int i = e / kBlock, j = e % kBlock;
            Am[i * LA + j] = j < i ? bet[i] * expf(gam[i] - gam[j]) * KK[i * LA + j] : 0.f;
        }
        if (t < D) {
            conv_ch(rawv, t, 2 * nq + (int64_t)h * D + t, X + D, LX, bet);
        } else if (t < 2 * D) {
            const int c = t - D;
            for (int i = 0; i < kBlock; ++i) X[i * LX + c] = (bet[i] * expf(gam[i])) * Yk[i * LQ + c];
        }
        __syncthreads();
        // P (overwrites the raw v tile) and the forward substitution (I + A) X = rhs
        for (int e = t; e < kBlock * kBlock; e += kThreads) {
            const int i = e / kBlock, j = e % kBlock;
            Ps[i * LP + j] = j <= i ? QK[i * LA + j] * expf(gam[i] - gam[j]) : 0.f;
        }
        if (t < 2 * D) {
            const int c = t;
            for (int i = 1; i < kBlock; ++i) {
                float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
                int j = 0;
                for (; j + 4 <= i; j += 4) {
                    a0 = fmaf(Am[i * LA + j], X[j * LX + c], a0);
                    a1 = fmaf(Am[i * LA + j + 1], X[(j + 1) * LX + c], a1);
                    a2 = fmaf(Am[i * LA + j + 2], X[(j + 2) * LX + c], a2);
                    a3 = fmaf(Am[i * LA + j + 3], X[(j + 3) * LX + c], a3);
                }
                for (; j < i; ++j) a0 = fmaf(Am[i * LA + j], X[j * LX + c], a0);
                X[i * LX + c] -= (a0 + a1) + (a2 + a3);
            }
        }
        __syncthreads();

        float *rec = p.ws_wu + ((int64_t)blk * Hv + h) * rec_floats(D);
        // Qe = e^gamma Q_hat - P W and O_intra = P U: warp w owns n-tiles [w*NT, w*NT + NT) of both
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
                    bw[nt][0] = tf32_bits(X[(8 * kk + t4) * LX + n0]);
                    bw[nt][1] = tf32_bits(X[(8 * kk + t4 + 4) * LX + n0]);
                    bu[nt][0] = tf32_bits(X[(8 * kk + t4) * LX + D + n0]);
                    bu[nt][1] = tf32_bits(X[(8 * kk + t4 + 4) * LX + D + n0]);
                }
#pragma unroll
                for (int mi = 0; mi < 4; ++mi) {
                    if (mi < kk / 2) continue;  // P is lower triangular
                    const float *pa = Ps + (16 * mi + g8) * LP + 8 * kk + t4;
                    const uint32_t a[4] = {tf32_bits(pa[0]), tf32_bits(pa[8 * LP]), tf32_bits(pa[4]),
                                           tf32_bits(pa[8 * LP + 4])};
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        mma_tf32(aq[mi][nt], a, bw[nt]);
                        mma_tf32(ao[mi][nt], a, bu[nt]);
                    }
                }
            }
            float *Qe = rec + kBlock * D, *Oi = rec + 4 * kBlock * D;
#pragma unroll
            for (int mi = 0; mi < 4; ++mi)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int c = (warp * NT + nt) * 8 + 2 * t4;
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        const int i = 16 * mi + g8 + 8 * hh;
                        const float e = eg[i];
                        float2 q2, o2;
                        q2.x = tf32_round(e * Yq[i * LQ + c] - aq[mi][nt][2 * hh]);
                        q2.y = tf32_round(e * Yq[i * LQ + c + 1] - aq[mi][nt][2 * hh + 1]);
                        o2.x = ao[mi][nt][2 * hh];
                        o2.y = ao[mi][nt][2 * hh + 1];
                        *reinterpret_cast<float2 *>(&Qe[i * D + c]) = q2;
                        *reinterpret_cast<float2 *>(&Oi[i * D + c]) = o2;
                    }
                }
        }
        // W (tf32), K_tilde (tf32), U (fp32), e^{gamma_63}
        {
            const float gl = gam[kBlock - 1];
            float *W = rec, *Kt = rec + 2 * kBlock * D, *U = rec + 3 * kBlock * D;
            for (int e = t; e < kBlock * D / 4; e += kThreads) {
                const int i = e / (D / 4), c = (e % (D / 4)) * 4;
                const float4 xw = *reinterpret_cast<const float4 *>(&X[i * LX + c]);
                const float4 xu = *reinterpret_cast<const float4 *>(&X[i * LX + D + c]);
                const float4 kk = *reinterpret_cast<const float4 *>(&Yk[i * LQ + c]);
                const float dj = expf(gl - gam[i]);
                *reinterpret_cast<float4 *>(&W[i * D + c]) =
                    make_float4(tf32_round(xw.x), tf32_round(xw.y), tf32_round(xw.z), tf32_round(xw.w));
                *reinterpret_cast<float4 *>(&Kt[i * D + c]) = make_float4(
                    tf32_round(dj * kk.x), tf32_round(dj * kk.y), tf32_round(dj * kk.z), tf32_round(dj * kk.w));
                *reinterpret_cast<float4 *>(&U[i * D + c]) = xu;
            }
            if (t == 0) rec[5 * kBlock * D] = expf(gl);
        }
    }
}

template <int D>
static cudaError_t launch(const LaunchCommon &p, int64_t ch, cudaStream_t st) {
    constexpr int LQ = D + 4, LA = kBlock + 1, LX = 2 * D + 8, LP = kBlock + 4;
    constexpr size_t smem =
        sizeof(float) * (2 * kBlock * LQ + 3 * kBlock * LA + kBlock * LX + kBlock * LP + 3 * kBlock);
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
