// Inter-block state pass and output, one CTA per (session, v-head, 16-column
// slice of d_v). Rows of S^T's columns are independent given the block
// factors, so the d_v split needs no exchange. Each CTA keeps its fp32 slice
// of S^T in shared memory and walks the session's blocks strictly in position
// order, so the result depends only on absolute positions:
//   U' = U - W S^T
//   O  = diag(exp(gamma)) Q_hat S^T + P U'
//   S^T <- exp(gamma_63) S^T + K_hat^T diag(exp(gamma_63 - gamma_j)) U'
#include "common.cuh"

namespace gdn {

constexpr int kSlice = 16;

template <int D>
__global__ void __launch_bounds__(kThreads, 1) state_kernel(const LaunchCommon p) {
    extern __shared__ __align__(16) float smem[];
    constexpr int LD = D + 4, LP = kBlock + 1, DS = kSlice;
    float *St = smem;                 // [D][DS]
    float *Ws = St + D * DS;          // [64][LD]
    float *Qs = Ws + kBlock * LD;     // [64][LD]
    float *Ks = Qs + kBlock * LD;     // [64][LD]
    float *Ps = Ks + kBlock * LD;     // [64][LP]
    float *Us = Ps + kBlock * LP;     // [64][DS]
    float *Up = Us + kBlock * DS;     // [64][DS]
    float *UD = Up + kBlock * DS;     // [64][DS]
    float *gs = UD + kBlock * DS;     // [64]

    constexpr int nsl = D / DS;
    const int sl = blockIdx.x % nsl;
    const int h = (blockIdx.x / nsl) % p.Hv;
    const int si = blockIdx.x / (nsl * p.Hv);
    const SessRef s = p.s[si];
    const int hk = h / p.G, c0 = sl * DS, t = threadIdx.x;
    const int Hv = p.Hv;

    float *Sg = s.S + (int64_t)h * D * D;
    const float *Sg0 = s.S0 + (int64_t)h * D * D;   // the starting state (the session's own, or a prefix's)
    for (int e = t; e < D * DS; e += kThreads) St[e] = Sg0[(e / DS) * D + c0 + e % DS];

    const int c = t % DS, i0 = t / DS;   // rows i0 + 16 r (outputs), key rows i0 + 16 r (state)
    const int nb = (s.n + kBlock - 1) / kBlock;
    for (int b = 0; b < nb; ++b) {
        const int blk = s.blk0 + b;
        const int nrow = min(kBlock, s.n - b * kBlock);
        const float *qk = p.ws_qk + ((int64_t)blk * p.Hk + hk) * qk_floats(D);
        const float *wu = p.ws_wu + ((int64_t)blk * Hv + h) * wu_floats(D);
        __syncthreads();
        for (int e = t; e < kBlock * D / 4; e += kThreads) {
            const int i = e / (D / 4), c4 = (e % (D / 4)) * 4;
            *reinterpret_cast<float4 *>(&Ws[i * LD + c4]) = *reinterpret_cast<const float4 *>(&wu[i * D + c4]);
            *reinterpret_cast<float4 *>(&Qs[i * LD + c4]) = *reinterpret_cast<const float4 *>(&qk[i * D + c4]);
            *reinterpret_cast<float4 *>(&Ks[i * LD + c4]) =
                *reinterpret_cast<const float4 *>(&qk[kBlock * D + i * D + c4]);
        }
        for (int e = t; e < kBlock * kBlock; e += kThreads) Ps[(e / kBlock) * LP + e % kBlock] = wu[2 * kBlock * D + e];
        for (int e = t; e < kBlock * DS; e += kThreads) Us[e] = wu[kBlock * D + (e / DS) * D + c0 + e % DS];
        if (t < kBlock) gs[t] = wu[2 * kBlock * D + kBlock * kBlock + t];
        __syncthreads();

        // U' = U - W S^T and the inter-block output term Q_hat S^T
        float ou[4] = {0.f, 0.f, 0.f, 0.f}, oq[4] = {0.f, 0.f, 0.f, 0.f};
        for (int k = 0; k < D; k += 4) {
            const float s0 = St[k * DS + c], s1 = St[(k + 1) * DS + c];
            const float s2 = St[(k + 2) * DS + c], s3 = St[(k + 3) * DS + c];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int i = i0 + 16 * r;
                const float4 w = *reinterpret_cast<const float4 *>(&Ws[i * LD + k]);
                const float4 q = *reinterpret_cast<const float4 *>(&Qs[i * LD + k]);
                ou[r] = fmaf(w.x, s0, ou[r]); ou[r] = fmaf(w.y, s1, ou[r]);
                ou[r] = fmaf(w.z, s2, ou[r]); ou[r] = fmaf(w.w, s3, ou[r]);
                oq[r] = fmaf(q.x, s0, oq[r]); oq[r] = fmaf(q.y, s1, oq[r]);
                oq[r] = fmaf(q.z, s2, oq[r]); oq[r] = fmaf(q.w, s3, oq[r]);
            }
        }
        const float glast = gs[kBlock - 1];
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = i0 + 16 * r;
            const float up = Us[i * DS + c] - ou[r];
            Up[i * DS + c] = up;
            UD[i * DS + c] = up * expf(glast - gs[i]);
            oq[r] *= expf(gs[i]);
        }
        __syncthreads();

        // outputs: O_i = exp(gamma_i) q_i S^T + sum_{j<=i} P_ij U'_j
        const int64_t orow0 = s.row0 + (int64_t)b * kBlock;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const int i = i0 + 16 * r;
            float acc = oq[r];
            for (int j = 0; j <= i; ++j) acc = fmaf(Ps[i * LP + j], Up[j * DS + c], acc);
            if (i < nrow) {
                const int64_t o = ((orow0 + i) * Hv + h) * D + c0 + c;
                if (p.out_bf16) static_cast<__nv_bfloat16 *>(p.out)[o] = __float2bfloat16_rn(acc);
                else static_cast<float *>(p.out)[o] = acc;
            }
        }
        // state: S^T <- exp(gamma_63) S^T + K_hat^T (U' scaled by exp(gamma_63 - gamma_j))
        const float eglast = expf(glast);
#pragma unroll
        for (int r = 0; r < D / 16; ++r) {
            const int k = i0 + 16 * r;
            float acc = 0.f;
            for (int j = 0; j < kBlock; ++j) acc = fmaf(Ks[j * LD + k], UD[j * DS + c], acc);
            St[k * DS + c] = fmaf(eglast, St[k * DS + c], acc);
        }
    }
    __syncthreads();
    for (int e = t; e < D * DS; e += kThreads) Sg[(e / DS) * D + c0 + e % DS] = St[e];
    if (s.S_cap) {   // the checkpoint of this call's final state
        float *Sc = s.S_cap + (int64_t)h * D * D;
        for (int e = t; e < D * DS; e += kThreads) Sc[(e / DS) * D + c0 + e % DS] = St[e];
    }
}

template <int D>
static cudaError_t launch(const LaunchCommon &p, cudaStream_t st) {
    constexpr int LD = D + 4, LP = kBlock + 1;
    constexpr size_t smem =
        sizeof(float) * (D * kSlice + 3 * kBlock * LD + kBlock * LP + 3 * kBlock * kSlice + kBlock);
    auto k = state_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<p.n_sess * p.Hv * (D / kSlice), kThreads, smem, st>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn

cudaError_t gdn_launch_state(const gdn::LaunchCommon &p, int D, cudaStream_t st) {
    return D == 64 ? gdn::launch<64>(p, st) : gdn::launch<128>(p, st);
}
