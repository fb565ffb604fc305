// Prologue + WY/UT transform, one CTA per (64-token block, q/k head).
//
// Per block, with the block's rows i = 0..63 (rows >= n are padding and are
// zero in every output):
//   causal conv (kernel 4) of the q, k, v channels, halo from the conv state
//   where the block starts a call; q_hat, k_hat = L2-normalised rows;
//   gamma_i = sum_{j<=i} g_j (cumulative log-decay inside the block);
//   A_ij = beta_i exp(gamma_i - gamma_j) k_hat_i . k_hat_j     (j < i)
//   (I + A) W = diag(beta exp(gamma)) K_hat,  (I + A) U = diag(beta) V
//   P_ij = exp(gamma_i - gamma_j) q_hat_i . k_hat_j             (j <= i)
// These are the intra-block factors of the chunked form of the gated delta
// rule S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T: with
// S0 the state before the block, U' = U - W S0^T, the outputs are
// O = diag(exp(gamma)) Q_hat S0^T + P U' and the next state is
// S^T = exp(gamma_63) S0^T + K_hat^T diag(exp(gamma_63 - gamma_j)) U'.
// Exponentials are taken of differences gamma_i - gamma_j <= 0 only, never
// factored into exp(gamma_i) exp(-gamma_j), so nothing overflows at any decay.
#include "common.cuh"

namespace gdn {

template <int D, typename InT>
__global__ void __launch_bounds__(kThreads, 1) prep_kernel(const LaunchCommon p, int64_t ch) {
    extern __shared__ __align__(16) float smem[];
    constexpr int LD = D + 4;       // row stride of q_hat / k_hat tiles
    constexpr int LX = 2 * D + 4;   // row stride of X = [W | U]
    constexpr int LA = kBlock + 1;  // row stride of 64x64 tiles
    float *Yq = smem;
    float *Yk = Yq + kBlock * LD;
    float *X = Yk + kBlock * LD;
    float *QK = X + kBlock * LX;
    float *KK = QK + kBlock * LA;
    float *Am = KK + kBlock * LA;
    float *gam = Am + kBlock * LA;
    float *bet = gam + kBlock;
    float *eg = bet + kBlock;

    const int blk = blockIdx.x, hk = blockIdx.y, t = threadIdx.x;
    const SessRef s = p.s[find_session(p, blk)];
    const int pos0 = (blk - s.blk0) * kBlock;     // block start, relative to the call's first token
    const int n = min(kBlock, s.n - pos0);         // valid rows
    const int64_t row0 = s.row0 + pos0;
    const int Hk = p.Hk, Hv = p.Hv;
    const int64_t nq = (int64_t)Hk * D, nv = (int64_t)Hv * D;
    const InT *cw = static_cast<const InT *>(p.conv_w);
    const InT *cs = static_cast<const InT *>(s.conv0);

    // 1. conv of the q and k channels of head hk (one channel per thread, sliding window)
    if (t < 2 * D) {
        const int which = t / D, c = t % D;
        const int64_t col = (int64_t)hk * D + c, chan = which * nq + col;
        const InT *x = static_cast<const InT *>(which ? p.xk : p.xq);
        float w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = to_f(cw[chan * 4 + i]);
        float h3, h2, h1;
        {
            float hv[3];
#pragma unroll
            for (int i = 0; i < 3; ++i) {
                const int pos = pos0 - 3 + i;
                hv[i] = pos >= 0 ? to_f(x[(s.row0 + pos) * nq + col]) : to_f(cs[(3 + pos) * ch + chan]);
            }
            h3 = hv[0]; h2 = hv[1]; h1 = hv[2];
        }
        float *Y = which ? Yk : Yq;
        for (int i = 0; i < kBlock; ++i) {
            const float x0 = i < n ? to_f(x[(row0 + i) * nq + col]) : 0.f;
            Y[i * LD + c] = conv_tap<InT>(w, h3, h2, h1, x0, p.act);
            h3 = h2; h2 = h1; h1 = x0;
        }
    }
    __syncthreads();

    // 2. L2 norm of each q and k row; padding rows become zero
    {
        const int warp = t >> 5, lane = t & 31;
        for (int r = warp; r < 2 * kBlock; r += kThreads / 32) {
            const int i = r % kBlock;
            float *row = (r < kBlock ? Yq : Yk) + i * LD;
            float ss = 0.f;
            for (int c = lane; c < D; c += 32) ss = fmaf(row[c], row[c], ss);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
            const float scale = (r < kBlock ? p.q_scale : 1.f) / sqrtf(ss + p.eps);
            for (int c = lane; c < D; c += 32) row[c] = i < n ? row[c] * scale : 0.f;
        }
    }
    __syncthreads();

    // q_hat, k_hat of this (block, k-head) to the workspace
    {
        float *wqk = p.ws_qk + ((int64_t)blk * Hk + hk) * qk_floats(D);
        constexpr int per = kBlock * D / 4;
        for (int e = t; e < 2 * per; e += kThreads) {
            const int which = e / per, rem = e % per, i = rem / (D / 4), c4 = rem % (D / 4);
            const float *Y = which ? Yk : Yq;
            *reinterpret_cast<float4 *>(&wqk[which * kBlock * D + i * D + c4 * 4]) =
                *reinterpret_cast<const float4 *>(&Y[i * LD + c4 * 4]);
        }
    }

    // 3. Q K^T (j <= i) and K K^T (j < i) in 4x4 register tiles
    {
        const int ti = t / 16, tj = t % 16;
        if (tj <= ti) {
            float aq[4][4], ak[4][4];
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) aq[a][b] = ak[a][b] = 0.f;
            for (int d = 0; d < D; d += 4) {
                float4 qi[4], ki[4], kj[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) {
                    qi[a] = *reinterpret_cast<const float4 *>(&Yq[(4 * ti + a) * LD + d]);
                    ki[a] = *reinterpret_cast<const float4 *>(&Yk[(4 * ti + a) * LD + d]);
                    kj[a] = *reinterpret_cast<const float4 *>(&Yk[(4 * tj + a) * LD + d]);
                }
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        aq[a][b] = fmaf(qi[a].x, kj[b].x, aq[a][b]);
                        aq[a][b] = fmaf(qi[a].y, kj[b].y, aq[a][b]);
                        aq[a][b] = fmaf(qi[a].z, kj[b].z, aq[a][b]);
                        aq[a][b] = fmaf(qi[a].w, kj[b].w, aq[a][b]);
                        ak[a][b] = fmaf(ki[a].x, kj[b].x, ak[a][b]);
                        ak[a][b] = fmaf(ki[a].y, kj[b].y, ak[a][b]);
                        ak[a][b] = fmaf(ki[a].z, kj[b].z, ak[a][b]);
                        ak[a][b] = fmaf(ki[a].w, kj[b].w, ak[a][b]);
                    }
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int i = 4 * ti + a, j = 4 * tj + b;
                    QK[i * LA + j] = j <= i ? aq[a][b] : 0.f;
                    KK[i * LA + j] = j < i ? ak[a][b] : 0.f;
                }
        }
    }

    // 4. per v-head of this group: gamma, A, forward substitution, W, U, P
    for (int gi = 0; gi < p.G; ++gi) {
        const int h = hk * p.G + gi;
        __syncthreads();
        if (t == 0) {
            float acc = 0.f;
            for (int i = 0; i < kBlock; ++i) {
                const bool valid = i < n;
                acc += valid ? p.g[(row0 + i) * Hv + h] : 0.f;
                gam[i] = acc;
                bet[i] = valid ? p.beta[(row0 + i) * Hv + h] : 0.f;
            }
        }
        __syncthreads();
        if (t < kBlock) eg[t] = expf(gam[t]);
        for (int e = t; e < kBlock * kBlock; e += kThreads) {
            const int i = e / kBlock, j = e % kBlock;
            Am[i * LA + j] = j < i ? bet[i] * expf(gam[i] - gam[j]) * KK[i * LA + j] : 0.f;
        }
        __syncthreads();
        // right-hand sides: X[:, 0:D] = beta e^gamma k_hat, X[:, D:2D] = beta v
        if (t < D) {
            const int c = t;
            const int64_t col = (int64_t)h * D + c, chan = 2 * nq + col;
            const InT *x = static_cast<const InT *>(p.xv);
            float w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) w[i] = to_f(cw[chan * 4 + i]);
            float hv[3];
#pragma unroll
            for (int i = 0; i < 3; ++i) {
                const int pos = pos0 - 3 + i;
                hv[i] = pos >= 0 ? to_f(x[(s.row0 + pos) * nv + col]) : to_f(cs[(3 + pos) * ch + chan]);
            }
            float h3 = hv[0], h2 = hv[1], h1 = hv[2];
            for (int i = 0; i < kBlock; ++i) {
                const float x0 = i < n ? to_f(x[(row0 + i) * nv + col]) : 0.f;
                const float y = conv_tap<InT>(w, h3, h2, h1, x0, p.act);
                X[i * LX + D + c] = i < n ? bet[i] * y : 0.f;
                h3 = h2; h2 = h1; h1 = x0;
            }
        } else if (t < 2 * D) {
            const int c = t - D;
            for (int i = 0; i < kBlock; ++i) X[i * LX + c] = (bet[i] * eg[i]) * Yk[i * LD + c];
        }
        __syncthreads();
        // (I + A) X = rhs by forward substitution, one column per thread
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
        float *wu = p.ws_wu + ((int64_t)blk * Hv + h) * wu_floats(D);
        constexpr int per = kBlock * D / 4;
        for (int e = t; e < 2 * per; e += kThreads) {
            const int which = e / per, rem = e % per, i = rem / (D / 4), c4 = rem % (D / 4);
            *reinterpret_cast<float4 *>(&wu[which * kBlock * D + i * D + c4 * 4]) =
                *reinterpret_cast<const float4 *>(&X[i * LX + which * D + c4 * 4]);
        }
        float *P = wu + 2 * kBlock * D;
        for (int e = t; e < kBlock * kBlock; e += kThreads) {
            const int i = e / kBlock, j = e % kBlock;
            P[e] = j <= i ? QK[i * LA + j] * expf(gam[i] - gam[j]) : 0.f;
        }
        if (t < kBlock) P[kBlock * kBlock + t] = gam[t];
    }
}

template <int D, typename InT>
static cudaError_t launch(const LaunchCommon &p, int64_t ch, cudaStream_t st) {
    constexpr int LD = D + 4, LX = 2 * D + 4, LA = kBlock + 1;
    constexpr size_t smem = sizeof(float) * (2 * kBlock * LD + kBlock * LX + 3 * kBlock * LA + 3 * kBlock);
    auto k = prep_kernel<D, InT>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<dim3(p.nblk, p.Hk), kThreads, smem, st>>>(p, ch);
    return cudaGetLastError();
}

}  // namespace gdn

cudaError_t gdn_launch_prep(const gdn::LaunchCommon &p, int D, int in_bf16, int64_t ch, cudaStream_t st) {
    using namespace gdn;
    if (D == 64) return in_bf16 ? launch<64, __nv_bfloat16>(p, ch, st) : launch<64, float>(p, ch, st);
    return in_bf16 ? launch<128, __nv_bfloat16>(p, ch, st) : launch<128, float>(p, ch, st);
}
