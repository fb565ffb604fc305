// Sequential state pass and outputs on tensor cores (bf16-input path): one CTA
// per (session, v-head, 16-column slice of d_v), 8 warps, walking the
// session's 64-token blocks strictly in position order. Per block, with the
// fp32 state slice S^T [D][16] in shared memory:
//   Z = [W; Qe] S^T                  (128 x 16; warp w owns rows 16w..16w+15)
//   U' = U - Z[0:64],  O = Z[64:128] + O_intra   (outputs written here)
//   S^T <- e^{gamma_63} S^T + K_tilde^T U'        (warp w owns state rows 16w..16w+15)
// Operands are tf32 (pre-rounded by the prologue, or rounded here for S^T and
// U'), accumulation is fp32, and the state itself stays fp32. The prologue
// stores each block's operands in fragment order, so one block is one
// contiguous copy; a two-stage cp.async pipeline fetches block b+1 while
// block b is computed. The CTA also commits its share of the session's conv
// state (nothing in this kernel reads it).
#include "common.cuh"
#include "mma.cuh"

namespace gdn {

template <int D>
__global__ void __launch_bounds__(kThreads, 1) chain_tc_kernel(const LaunchCommon p, int64_t ch) {
    extern __shared__ __align__(16) float smem[];
    constexpr int DS = kSliceCols, NT = DS / 8;
    constexpr int SP = DS + 8;                 // S^T and U' rows (B fragments): banks 24t + g, distinct
    constexpr int WQF = 2 * kBlock * D;        // [W; Qe] fragments
    constexpr int KTF = kBlock * D;            // K_tilde^T fragments
    constexpr int UF = kBlock * DS;            // one slice of U (or O_intra) fragments
    constexpr int STAGE = WQF + KTF + 2 * UF + 4;
    static_assert(D == 128 || D == 64, "head dim");
    float *St = smem + 2 * STAGE;              // [D][SP]   fp32 state slice
    float *Ups = St + D * SP;                  // [64][SP]  tf32 U'

    constexpr int nsl = D / DS;
    const int sl = blockIdx.x % nsl;
    const int h = (blockIdx.x / nsl) % p.Hv;
    const int si = blockIdx.x / (nsl * p.Hv);
    const SessRef s = p.s[si];
    const int c0 = sl * DS, t = threadIdx.x, warp = t >> 5, lane = t & 31, g8 = lane >> 2, t4 = lane & 3;
    const int Hv = p.Hv;
    const int nb = (s.n + kBlock - 1) / kBlock;
    const int64_t RF = rec_floats(D);

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
            const __nv_bfloat16 o0 = cs[chan], o1 = cs[ch + chan], o2 = cs[2 * ch + chan];
            __nv_bfloat16 nw[3];
#pragma unroll
            for (int r = 0; r < 3; ++r) {
                const int pos = s.n - 3 + r;
                nw[r] = pos >= 0 ? x[(s.row0 + pos) * ld + col] : (pos == -3 ? o0 : (pos == -2 ? o1 : o2));
            }
#pragma unroll
            for (int r = 0; r < 3; ++r) cs[r * ch + chan] = nw[r];
        }
    }

    auto issue = [&](int b) {
        float *buf = smem + (b & 1) * STAGE;
        const float *r = p.ws_wu + ((int64_t)(s.blk0 + b) * Hv + h) * RF;
        for (int e = t; e < (WQF + KTF) / 4; e += kThreads) cp_async16(buf + 4 * e, r + 4 * e);
        for (int e = t; e < 2 * UF / 4; e += kThreads) {
            const int which = e / (UF / 4), q = e % (UF / 4);
            cp_async16(buf + WQF + KTF + which * UF + 4 * q, r + (192 + 64 * which) * D + sl * UF + 4 * q);
        }
        if (t == 0) cp_async16(buf + WQF + KTF + 2 * UF, r + 320 * D);
    };

    float *Sg = s.S + (int64_t)h * D * D;
    for (int e = t; e < D * DS; e += kThreads) St[(e / DS) * SP + e % DS] = Sg[(int64_t)(e / DS) * D + c0 + e % DS];
    if (nb > 0) issue(0);
    cp_async_commit();

    for (int b = 0; b < nb; ++b) {
        const float *buf = smem + (b & 1) * STAGE;
        if (b + 1 < nb) issue(b + 1);   // the other stage was released at the end of step b-1
        cp_async_commit();
        cp_async_wait<1>();             // block b's group has landed (this thread's part)
        __syncthreads();                // (A) ... and everyone's

        // Z = [W; Qe] S^T, two partial accumulators (even / odd k-steps) per n-tile
        float acc[NT][4], acc2[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int f = 0; f < 4; ++f) acc[nt][f] = acc2[nt][f] = 0.f;
        {
            const float4 *wa = reinterpret_cast<const float4 *>(buf) + (warp * (D / 8)) * 32 + lane;
#pragma unroll
            for (int ks = 0; ks < D / 8; ++ks) {
                const float4 av = wa[ks * 32];
                const uint32_t a[4] = {__float_as_uint(av.x), __float_as_uint(av.y), __float_as_uint(av.z),
                                       __float_as_uint(av.w)};
                const int k0 = 8 * ks;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint32_t bb[2] = {tf32_bits(St[(k0 + t4) * SP + 8 * nt + g8]),
                                            tf32_bits(St[(k0 + t4 + 4) * SP + 8 * nt + g8])};
                    mma_tf32((ks & 1) ? acc2[nt] : acc[nt], a, bb);
                }
            }
        }
        // U' (warps 0-3) and outputs (warps 4-7); C fragments match the stored order
        {
            const int nrow = min(kBlock, s.n - b * kBlock);
            const int w4 = warp & 3;
            const float4 *uo = reinterpret_cast<const float4 *>(buf + WQF + KTF + (warp < 4 ? 0 : UF));
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const float4 u = uo[(w4 * NT + nt) * 32 + lane];
                const float z[4] = {acc[nt][0] + acc2[nt][0], acc[nt][1] + acc2[nt][1], acc[nt][2] + acc2[nt][2],
                                    acc[nt][3] + acc2[nt][3]};
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
        __syncthreads();  // (B) U' complete
        // S^T <- e^{gamma_63} S^T + K_tilde^T U'   (D / 16 warps own the state rows)
        if (16 * warp < D) {
            const float e = buf[WQF + KTF + 2 * UF];
            const int m0 = 16 * warp + g8;
            float cst[NT][4], cst2[NT][4];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int c = 8 * nt + 2 * t4;
                cst[nt][0] = e * St[m0 * SP + c];
                cst[nt][1] = e * St[m0 * SP + c + 1];
                cst[nt][2] = e * St[(m0 + 8) * SP + c];
                cst[nt][3] = e * St[(m0 + 8) * SP + c + 1];
#pragma unroll
                for (int f = 0; f < 4; ++f) cst2[nt][f] = 0.f;
            }
            const float4 *ka = reinterpret_cast<const float4 *>(buf + WQF) + (warp * 8) * 32 + lane;
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
                    mma_tf32((ks & 1) ? cst2[nt] : cst[nt], a, bb);
                }
            }
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int c = 8 * nt + 2 * t4;
                St[m0 * SP + c] = cst[nt][0] + cst2[nt][0];
                St[m0 * SP + c + 1] = cst[nt][1] + cst2[nt][1];
                St[(m0 + 8) * SP + c] = cst[nt][2] + cst2[nt][2];
                St[(m0 + 8) * SP + c + 1] = cst[nt][3] + cst2[nt][3];
            }
        }
        __syncthreads();  // (C) S^T updated; this stage is free for block b+2
    }
    cp_async_wait<0>();
    __syncthreads();
    for (int e = t; e < D * DS; e += kThreads) Sg[(int64_t)(e / DS) * D + c0 + e % DS] = St[(e / DS) * SP + e % DS];
}

template <int D>
static cudaError_t launch(const LaunchCommon &p, int64_t ch, cudaStream_t st) {
    constexpr int DS = kSliceCols, SP = DS + 8;
    constexpr size_t smem = sizeof(float) * (2 * (2 * kBlock * D + kBlock * D + 2 * kBlock * DS + 4) + D * SP +
                                             kBlock * SP);
    auto k = chain_tc_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<p.n_sess * p.Hv * (D / DS), kThreads, smem, st>>>(p, ch);
    return cudaGetLastError();
}

}  // namespace gdn

cudaError_t gdn_launch_chain_tc(const gdn::LaunchCommon &p, int D, int64_t ch, cudaStream_t st) {
    return D == 64 ? gdn::launch<64>(p, ch, st) : gdn::launch<128>(p, ch, st);
}
