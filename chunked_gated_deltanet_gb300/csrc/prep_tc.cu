// Prologue + WY/UT transform on the warp-level tensor-core path (mma.sync),
// bf16 inputs, d_k = d_v = 64 (d = 128 runs the tcgen05 prologue,
// prep_umma.cu). One CTA per (64-token block, q/k head), for each of the
// head's G v-heads.
//
// Per block (rows i = 0..63; rows >= n are padding and zero everywhere):
//   conv (kernel 4, halo from the conv state at a call's first block), L2 norm
//   gamma = cumulative log-decay in the block
//   Q K^T, K K^T                                    bf16x3 MMA (hi/lo split), lower triangle
//   A_ij = beta_i e^{gamma_i - gamma_j} (K K^T)_ij      (j < i)
//   T = (I + A)^{-1}                                 blocked 16 x 16 inverse, fp32
//   W = T diag(beta e^gamma) K_hat,  U = T diag(beta) V     split-tf32 MMA
//   P_ij = e^{gamma_i - gamma_j} (Q K^T)_ij              (j <= i)
//   Qe = diag(e^gamma) Q_hat - P W,  O_intra = P U          tf32 MMA
//   K_tilde = diag(e^{gamma_63 - gamma_j}) K_hat
// so that, with S0 the state entering the block, the outputs are
// O = Qe S0^T + O_intra and U' = U - W S0^T feeds S^T <- e^{gamma_63} S0^T + K_tilde^T U'.
// The record is written in the fragment order of the state kernel (see common.cuh).
// Conv and norm run one warp per row (each lane owns D/32 channels), so the
// norm's reduction is a single warp shuffle; every input tile is requested at
// kernel start.
#include "common.cuh"
#include "mma.cuh"

namespace gdn {

constexpr int kPrepThreads = 512;

template <int D>
__global__ void __launch_bounds__(kPrepThreads, 1) prep_tc_kernel(const LaunchCommon p, int64_t ch) {
    extern __shared__ __align__(16) float smem[];
    constexpr int LQ = D + 4;       // q_hat / k_hat fp32 rows
    constexpr int LA = kBlock + 1;  // Q K^T, K K^T
    constexpr int LT = kBlock + 4;  // T, A and P: row-indexed A fragments, banks 4g + t
    constexpr int LB = D + 8;       // fp32 B operands indexed [token][column]: banks 8t + g
    constexpr int LH = D + 8;       // bf16 hi/lo rows: 32-bit fragment words hit banks 4g + t
    constexpr int CPL = D / 32;     // channels per lane in the row-parallel conv
    constexpr int RAW = (kBlock + 3) * D;
    float *Yq = smem;
    float *Yk = Yq + kBlock * LQ;
    float *QK = Yk + kBlock * LQ;
    float *KK = QK + kBlock * LA;
    float *Tm = KK + kBlock * LA;
    float *Ps = Tm + kBlock * LT;   // raw v tile, then A during the inverse, then P
    float *Bk = Ps + kBlock * LT;   // bf16 q/k hi, then inverse scratch, then beta e^gamma k_hat, then W
    float *Bv = Bk + kBlock * LB;   // bf16 q/k lo, then beta v, then U
    float *gam = Bv + kBlock * LB;
    float *bet = gam + kBlock;
    float *egv = bet + kBlock;
    __nv_bfloat16 *rawq = reinterpret_cast<__nv_bfloat16 *>(QK);   // QK, KK, Tm are free at the start
    __nv_bfloat16 *rawk = rawq + RAW;
    __nv_bfloat16 *rawv = reinterpret_cast<__nv_bfloat16 *>(Ps);
    __nv_bfloat16 *Qh = reinterpret_cast<__nv_bfloat16 *>(Bk), *Kh = Qh + kBlock * LH;
    __nv_bfloat16 *Ql = reinterpret_cast<__nv_bfloat16 *>(Bv), *Kl = Ql + kBlock * LH;
    float *Mt = Bk;                 // 3 x 16 x 17 inverse scratch (the hi/lo arrays are dead by then)
    static_assert(2 * RAW * 2 <= (2 * kBlock * LA + kBlock * LT) * 4, "q/k raw tiles must fit QK, KK, T");
    static_assert(RAW * 2 <= kBlock * LT * 4, "v raw tile must fit the P region");
    static_assert(2 * kBlock * LH * 2 <= kBlock * LB * 4, "hi (lo) arrays of q and k must fit one B region");

    const int blk = blockIdx.x, hk = blockIdx.y, t = threadIdx.x;
    const int warp = t >> 5, lane = t & 31, g8 = lane >> 2, t4 = lane & 3;
    const SessRef s = p.s[find_session(p, blk)];
    const int pos0 = (blk - s.blk0) * kBlock;
    const int n = min(kBlock, s.n - pos0);
    const int64_t row0 = s.row0 + pos0;
    const int Hk = p.Hk, Hv = p.Hv;
    const int64_t nq = (int64_t)Hk * D, nv = (int64_t)Hv * D;
    const __nv_bfloat16 *cw = static_cast<const __nv_bfloat16 *>(p.conv_w);
    const __nv_bfloat16 *cs = static_cast<const __nv_bfloat16 *>(s.conv0);

    // Stage rows pos0-3 .. pos0+63 of one head's channels; rows before the call
    // come from the conv state, rows past the block's valid rows are zero.
    auto stage = [&](__nv_bfloat16 *dst, const __nv_bfloat16 *x, int64_t ld, int64_t col0, int64_t chan0) {
        constexpr int CH = D / 8;
        for (int e = t; e < (kBlock + 3) * CH; e += kPrepThreads) {
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
    // Row-parallel conv of rows [r0, r0 + nr) of a staged tile: lane owns channels lane*CPL ..
    // Rows go four at a time so that four independent chains are in flight;
    // the outputs go through `emit(i, y[CPL])`.
    auto load_row = [&](const __nv_bfloat16 *raw, int r, float (&v)[CPL]) {
        if constexpr (CPL == 4) {
            const uint2 u = *reinterpret_cast<const uint2 *>(raw + r * D + lane * 4);
            const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(&u.x);
            const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162 *>(&u.y);
            v[0] = __low2float(a); v[1] = __high2float(a); v[2] = __low2float(b); v[3] = __high2float(b);
        } else {
            const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162 *>(raw + r * D + lane * 2);
            v[0] = __low2float(a); v[1] = __high2float(a);
        }
    };
    auto conv_rows = [&](const __nv_bfloat16 *raw, int64_t chan0, int r0, int nr, auto &&emit) {
        float w[CPL][4];
#pragma unroll
        for (int c = 0; c < CPL; ++c)
#pragma unroll
            for (int k = 0; k < 4; ++k) w[c][k] = __bfloat162float(cw[(chan0 + lane * CPL + c) * 4 + k]);
        for (int i0 = r0; i0 < r0 + nr; i0 += 4) {
            float x[7][CPL];   // raw rows i0 .. i0+6 = block rows i0-3 .. i0+3
#pragma unroll
            for (int r = 0; r < 7; ++r) load_row(raw, i0 + r, x[r]);
            float y[4][CPL];
#pragma unroll
            for (int u = 0; u < 4; ++u)
#pragma unroll
                for (int c = 0; c < CPL; ++c)
                    y[u][c] = conv_tap<__nv_bfloat16>(w[c], x[u][c], x[u + 1][c], x[u + 2][c], x[u + 3][c], p.act);
            emit(i0, y);
        }
    };

    // 1. request every input tile; g and beta of the first v-head into registers
    stage(rawq, static_cast<const __nv_bfloat16 *>(p.xq), nq, (int64_t)hk * D, (int64_t)hk * D);
    stage(rawk, static_cast<const __nv_bfloat16 *>(p.xk), nq, (int64_t)hk * D, nq + (int64_t)hk * D);
    stage(rawv, static_cast<const __nv_bfloat16 *>(p.xv), nv, (int64_t)(hk * p.G) * D, 2 * nq + (int64_t)(hk * p.G) * D);
    float gv = 0.f, bv = 0.f;
    if (t < kBlock && t < n) {
        gv = p.g[(row0 + t) * Hv + hk * p.G];
        bv = p.beta[(row0 + t) * Hv + hk * p.G];
    }
    cp_async_wait<1>();   // q and k tiles (v may still be in flight)
    __syncthreads();

    // 2. conv + L2 norm of q (warps 0-7) and k (warps 8-15), 8 rows per warp; fp32 rows and bf16 hi/lo
    {
        const int which = warp >> 3;
        float *Y = which ? Yk : Yq;
        __nv_bfloat16 *Hh = which ? Kh : Qh, *Hl = which ? Kl : Ql;
        const float qs = which ? 1.f : p.q_scale;
        conv_rows(which ? rawk : rawq, which * nq + (int64_t)hk * D, 8 * (warp & 7), 8, [&](int i0, float (&y)[4][CPL]) {
            float ss[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                ss[u] = 0.f;
#pragma unroll
                for (int c = 0; c < CPL; ++c) ss[u] = fmaf(y[u][c], y[u][c], ss[u]);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1)
#pragma unroll
                for (int u = 0; u < 4; ++u) ss[u] += __shfl_xor_sync(0xffffffffu, ss[u], o);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u;
                const float scale = qs * rsqrtf(ss[u] + p.eps);
                float v[CPL];
                __nv_bfloat16 hi[CPL], lo[CPL];
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    v[c] = i < n ? y[u][c] * scale : 0.f;
                    split_bf16(v[c], hi[c], lo[c]);
                }
                if constexpr (CPL == 4) {
                    *reinterpret_cast<float4 *>(&Y[i * LQ + lane * 4]) = make_float4(v[0], v[1], v[2], v[3]);
                    *reinterpret_cast<uint2 *>(&Hh[i * LH + lane * 4]) =
                        make_uint2(pack_bf16(hi[0], hi[1]), pack_bf16(hi[2], hi[3]));
                    *reinterpret_cast<uint2 *>(&Hl[i * LH + lane * 4]) =
                        make_uint2(pack_bf16(lo[0], lo[1]), pack_bf16(lo[2], lo[3]));
                } else {
                    *reinterpret_cast<float2 *>(&Y[i * LQ + lane * 2]) = make_float2(v[0], v[1]);
                    *reinterpret_cast<uint32_t *>(&Hh[i * LH + lane * 2]) = pack_bf16(hi[0], hi[1]);
                    *reinterpret_cast<uint32_t *>(&Hl[i * LH + lane * 2]) = pack_bf16(lo[0], lo[1]);
                }
            }
        });
    }
    __syncthreads();

    // 3. Q K^T and K K^T on the 20 lower-triangle 16x8 tiles, bf16x3 (hi*hi + hi*lo + lo*hi):
    //    these dot products of unit vectors can cancel, and one rounding would show in short sequences
    for (int tile = warp; tile < 20; tile += kPrepThreads / 32) {
        int mi = 0, rem = tile;
        while (rem >= 2 * mi + 2) { rem -= 2 * mi + 2; ++mi; }
        const int nj = rem;
        float cq[4] = {0.f, 0.f, 0.f, 0.f}, ck[4] = {0.f, 0.f, 0.f, 0.f};
        float cq2[4] = {0.f, 0.f, 0.f, 0.f}, ck2[4] = {0.f, 0.f, 0.f, 0.f};
        auto word = [&](const __nv_bfloat16 *base, int row, int col) {
            return *reinterpret_cast<const uint32_t *>(base + row * LH + col);
        };
        const int ra = 16 * mi + g8, rb = 8 * nj + g8;
#pragma unroll
        for (int k0 = 0; k0 < D; k0 += 16) {
            const int ca = k0 + 2 * t4;
            const uint32_t aqh[4] = {word(Qh, ra, ca), word(Qh, ra + 8, ca), word(Qh, ra, ca + 8), word(Qh, ra + 8, ca + 8)};
            const uint32_t aql[4] = {word(Ql, ra, ca), word(Ql, ra + 8, ca), word(Ql, ra, ca + 8), word(Ql, ra + 8, ca + 8)};
            const uint32_t akh[4] = {word(Kh, ra, ca), word(Kh, ra + 8, ca), word(Kh, ra, ca + 8), word(Kh, ra + 8, ca + 8)};
            const uint32_t akl[4] = {word(Kl, ra, ca), word(Kl, ra + 8, ca), word(Kl, ra, ca + 8), word(Kl, ra + 8, ca + 8)};
            const uint32_t bh[2] = {word(Kh, rb, ca), word(Kh, rb, ca + 8)};
            const uint32_t bl[2] = {word(Kl, rb, ca), word(Kl, rb, ca + 8)};
            float(&q1)[4] = (k0 & 16) ? cq2 : cq;
            float(&k1)[4] = (k0 & 16) ? ck2 : ck;
            mma_bf16(q1, aql, bh);
            mma_bf16(q1, aqh, bl);
            mma_bf16(q1, aqh, bh);
            mma_bf16(k1, akl, bh);
            mma_bf16(k1, akh, bl);
            mma_bf16(k1, akh, bh);
        }
        const int i0 = 16 * mi + g8, j0 = 8 * nj + 2 * t4;
        QK[i0 * LA + j0] = cq[0] + cq2[0]; QK[i0 * LA + j0 + 1] = cq[1] + cq2[1];
        QK[(i0 + 8) * LA + j0] = cq[2] + cq2[2]; QK[(i0 + 8) * LA + j0 + 1] = cq[3] + cq2[3];
        KK[i0 * LA + j0] = ck[0] + ck2[0]; KK[i0 * LA + j0 + 1] = ck[1] + ck2[1];
        KK[(i0 + 8) * LA + j0] = ck[2] + ck2[2]; KK[(i0 + 8) * LA + j0 + 1] = ck[3] + ck2[3];
    }

    // 4. each v-head of the group
    for (int gi = 0; gi < p.G; ++gi) {
        const int h = hk * p.G + gi;
        if (gi > 0) {      // the first head's g, beta and v tile were requested at kernel start
            __syncthreads();   // the previous head is done with the P region
            stage(rawv, static_cast<const __nv_bfloat16 *>(p.xv), nv, (int64_t)h * D, 2 * nq + (int64_t)h * D);
            gv = bv = 0.f;
            if (t < kBlock && t < n) {
                gv = p.g[(row0 + t) * Hv + h];
                bv = p.beta[(row0 + t) * Hv + h];
            }
        }
        if (t < kBlock) {   // gamma: inclusive scan of g (two warps)
            float sv = gv;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, sv, o);
                if (lane >= o) sv += y;
            }
            gam[t] = sv;
            bet[t] = bv;
        }
        cp_async_wait<0>();
        __syncthreads();   // QK/KK, v tile, warp scans
        if (t >= 32 && t < kBlock) gam[t] += gam[31];
        __syncthreads();
        if (t < kBlock) egv[t] = expf(gam[t]);
        // beta v (row-parallel conv, 8 rows per warp) into Bv; A (strict lower) into the P region later
        conv_rows(rawv, 2 * nq + (int64_t)h * D, 4 * warp, 4, [&](int i0, float (&y)[4][CPL]) {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = i0 + u;
                const float b = i < n ? bet[i] : 0.f;
#pragma unroll
                for (int c = 0; c < CPL; ++c) Bv[i * LB + lane * CPL + c] = b * y[u][c];
            }
        });
        __syncthreads();   // the raw v tile is consumed
        for (int e = t; e < kBlock * kBlock; e += kPrepThreads) {
            const int i = e / kBlock, j = e % kBlock;
            Ps[i * LT + j] = j < i ? bet[i] * expf(gam[i] - gam[j]) * KK[i * LA + j] : 0.f;
        }
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
            for (int e = t; e < nblkd * 256; e += kPrepThreads) {
                const int jb = e >> 8, r = (e >> 4) & 15, c = e & 15, ib = jb + dist;
                float sum = 0.f;
                for (int k = 16 * jb; k < 16 * ib; ++k) sum = fmaf(Ps[(16 * ib + r) * LT + k], Tm[k * LT + 16 * jb + c], sum);
                Mt[(jb * 16 + r) * 17 + c] = sum;
            }
            __syncthreads();
            for (int e = t; e < nblkd * 256; e += kPrepThreads) {
                const int jb = e >> 8, r = (e >> 4) & 15, c = e & 15, ib = jb + dist;
                float sum = 0.f;
#pragma unroll
                for (int k = 0; k < 16; ++k) sum = fmaf(Tm[(16 * ib + r) * LT + 16 * ib + k], Mt[(jb * 16 + k) * 17 + c], sum);
                Tm[(16 * ib + r) * LT + 16 * jb + c] = -sum;
            }
            __syncthreads();
        }
        // B operand beta e^gamma k_hat (over the scratch); P over A
        for (int e = t; e < kBlock * D; e += kPrepThreads) {
            const int i = e / D, c = e % D;
            Bk[i * LB + c] = (bet[i] * egv[i]) * Yk[i * LQ + c];
        }
        for (int e = t; e < kBlock * kBlock; e += kPrepThreads) {
            const int i = e / kBlock, j = e % kBlock;
            Ps[i * LT + j] = j <= i ? QK[i * LA + j] * expf(gam[i] - gam[j]) : 0.f;
        }
        __syncthreads();

        float *rec = p.ws_wu + ((int64_t)blk * Hv + h) * rec_floats(D);
        // W = T Bk (warps 0-3) and U = T Bv (warps 4-7), split tf32, T lower triangular
        {
            constexpr int NW = D / 64;   // n-tiles per warp
            const float *B = warp < 8 ? Bk : Bv;
            const int nbase = (warp & 7) * NW * 8;
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
            float *dst = warp < 8 ? Bk : Bv;
#pragma unroll
            for (int mi = 0; mi < 4; ++mi)
#pragma unroll
                for (int nt = 0; nt < NW; ++nt) {
                    const int c = nbase + nt * 8 + 2 * t4, i = 16 * mi + g8;
                    dst[i * LB + c] = acc[mi][nt][0];
                    dst[i * LB + c + 1] = acc[mi][nt][1];
                    dst[(i + 8) * LB + c] = acc[mi][nt][2];
                    dst[(i + 8) * LB + c + 1] = acc[mi][nt][3];
                    if (warp >= 8)   // U goes out as-is, in C-fragment slice order
                        *reinterpret_cast<float4 *>(rec + 192 * D + cfrag_slice_index(i, c)) =
                            make_float4(acc[mi][nt][0], acc[mi][nt][1], acc[mi][nt][2], acc[mi][nt][3]);
                }
        }
        __syncthreads();

        // Qe = e^gamma Q_hat - P W (warps 0-7) and O_intra = P U (warps 8-15), tf32; warp owns D/64 n-tiles
        {
            constexpr int NT = D / 64;
            const bool isq = warp < 8;
            const float *B = isq ? Bk : Bv;
            const int nb0 = (warp & 7) * NT * 8;
            float ac[4][NT][4];
#pragma unroll
            for (int mi = 0; mi < 4; ++mi)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int f = 0; f < 4; ++f) ac[mi][nt][f] = 0.f;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                uint32_t bw[NT][2];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int n0 = nb0 + nt * 8 + g8;
                    bw[nt][0] = tf32_bits(B[(8 * kk + t4) * LB + n0]);
                    bw[nt][1] = tf32_bits(B[(8 * kk + t4 + 4) * LB + n0]);
                }
#pragma unroll
                for (int mi = 0; mi < 4; ++mi) {
                    if (mi < kk / 2) continue;  // P is lower triangular
                    const float *pa = Ps + (16 * mi + g8) * LT + 8 * kk + t4;
                    const uint32_t a[4] = {tf32_bits(pa[0]), tf32_bits(pa[8 * LT]), tf32_bits(pa[4]),
                                           tf32_bits(pa[8 * LT + 4])};
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) mma_tf32(ac[mi][nt], a, bw[nt]);
                }
            }
#pragma unroll
            for (int mi = 0; mi < 4; ++mi)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int c = nb0 + nt * 8 + 2 * t4, i = 16 * mi + g8;
                    if (!isq) {
                        *reinterpret_cast<float4 *>(rec + 256 * D + cfrag_slice_index(i, c)) =
                            make_float4(ac[mi][nt][0], ac[mi][nt][1], ac[mi][nt][2], ac[mi][nt][3]);
                    } else {
#pragma unroll
                        for (int f = 0; f < 4; ++f) {
                            const int ii = i + 8 * (f >> 1), cc = c + (f & 1);
                            rec[afrag_index(kBlock + ii, cc, D)] =
                                tf32_round(egv[ii] * Yq[ii * LQ + cc] - ac[mi][nt][f]);
                        }
                    }
                }
        }
        // W (rows 0..63 of [W; Qe]) and K_tilde^T as A fragments, tf32; e^{gamma_63}
        {
            const float gl = gam[kBlock - 1];
            constexpr int NW4 = 4 * (D / 8) * 32;   // float4 groups of W
            for (int e = t; e < NW4 + (D / 16) * 8 * 32; e += kPrepThreads) {
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
    k<<<dim3(p.nblk, p.Hk), kPrepThreads, smem, st>>>(p, ch);
    return cudaGetLastError();
}

}  // namespace gdn

cudaError_t gdn_launch_prep_tc(const gdn::LaunchCommon &p, int D, int64_t ch, cudaStream_t st) {
    if (D != 64) return cudaErrorInvalidValue;   // d = 128 has its own prologue
    return gdn::launch<64>(p, ch, st);
}
