// Sequential state pass and outputs on tensor cores (bf16-input path): one CTA
// per (session, v-head, DS-column slice of d_v), 8 warps, walking the
// session's 64-token blocks strictly in position order. Per block, with the
// fp32 state slice S^T [D][DS] in shared memory:
//   Z = [W; Qe] S^T                  (128 x DS; warp w owns rows 16w..16w+15)
//   U' = U - Z[0:64],  O = Z[64:128] + O_intra   (outputs written here)
//   S^T <- e^{gamma_63} S^T + K_tilde^T U'        (warp w owns state rows 16w..16w+15)
// Operands are tf32 (pre-rounded by the prologue, or rounded here for S^T and
// U'), accumulation is fp32, and the state itself stays fp32. The next block's
// [W; Qe] is fetched with cp.async while the current block's state update
// runs, and its K_tilde, U, O_intra while the next [W; Qe] product runs.
#include "common.cuh"
#include "mma.cuh"

namespace gdn {

template <int D, int DS>
__global__ void __launch_bounds__(kThreads, 1) chain_tc_kernel(const LaunchCommon p) {
    extern __shared__ __align__(16) float smem[];
    constexpr int LW = D + 4;                    // [W; Qe] rows: A fragments, banks 4g + t
    constexpr int LK = D + 8;                    // K_tilde rows read transposed: banks 8t + g
    constexpr int SP = DS == 8 ? 8 : DS + 8;     // S^T and U' rows (B fragments): banks 8t + g or 24t + g
    constexpr int NT = DS / 8;
    static_assert(D == 128 || D == 64, "head dim");
    float *WQs = smem;                  // [2*64][LW]
    float *Kts = WQs + 2 * kBlock * LW;  // [64][LK]
    float *St = Kts + kBlock * LK;       // [D][SP]   fp32 state slice
    float *Ups = St + D * SP;            // [64][SP]  tf32 U'
    float *Us = Ups + kBlock * SP;       // [64][DS]
    float *Ois = Us + kBlock * DS;       // [64][DS]
    float *egs = Ois + kBlock * DS;      // [4]

    constexpr int nsl = D / DS;
    const int sl = blockIdx.x % nsl;
    const int h = (blockIdx.x / nsl) % p.Hv;
    const int si = blockIdx.x / (nsl * p.Hv);
    const SessRef s = p.s[si];
    const int c0 = sl * DS, t = threadIdx.x, warp = t >> 5, lane = t & 31, g8 = lane >> 2, t4 = lane & 3;
    const int Hv = p.Hv;
    const int nb = (s.n + kBlock - 1) / kBlock;
    const int64_t RF = rec_floats(D);

    auto rec_of = [&](int b) { return p.ws_wu + ((int64_t)(s.blk0 + b) * Hv + h) * RF; };
    auto load_wq = [&](int b) {
        const float *r = rec_of(b);
        for (int e = t; e < 2 * kBlock * D / 4; e += kThreads) {
            const int i = e / (D / 4), c = (e % (D / 4)) * 4;
            cp_async16(&WQs[i * LW + c], r + (int64_t)i * D + c);
        }
    };
    auto load_rest = [&](int b) {
        const float *r = rec_of(b);
        for (int e = t; e < kBlock * D / 4; e += kThreads) {
            const int i = e / (D / 4), c = (e % (D / 4)) * 4;
            cp_async16(&Kts[i * LK + c], r + 2 * kBlock * D + (int64_t)i * D + c);
        }
        for (int e = t; e < 2 * kBlock * DS / 4; e += kThreads) {
            const int which = e / (kBlock * DS / 4), rem = e % (kBlock * DS / 4);
            const int i = rem / (DS / 4), c = (rem % (DS / 4)) * 4;
            cp_async16((which ? Ois : Us) + i * DS + c, r + (3 + which) * kBlock * D + (int64_t)i * D + c0 + c);
        }
        if (t == 0) cp_async16(egs, r + 5 * kBlock * D);
    };

    // state slice in
    float *Sg = s.S + (int64_t)h * D * D;
    for (int e = t; e < D * DS; e += kThreads) St[(e / DS) * SP + e % DS] = Sg[(int64_t)(e / DS) * D + c0 + e % DS];
    if (nb > 0) {
        load_rest(0);
        cp_async_commit();
        load_wq(0);
        cp_async_commit();
    }
    cp_async_wait<0>();
    __syncthreads();

    for (int b = 0; b < nb; ++b) {
        // Z = [W; Qe] S^T, two partial accumulators (even / odd k-steps) per n-tile
        float acc[NT][4], acc2[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int f = 0; f < 4; ++f) acc[nt][f] = acc2[nt][f] = 0.f;
        {
            const float *wa = WQs + (16 * warp + g8) * LW + t4;
#pragma unroll
            for (int ks = 0; ks < D / 8; ++ks) {
                const int k0 = 8 * ks;
                const uint32_t a[4] = {__float_as_uint(wa[k0]), __float_as_uint(wa[8 * LW + k0]),
                                       __float_as_uint(wa[k0 + 4]), __float_as_uint(wa[8 * LW + k0 + 4])};
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const uint32_t bb[2] = {tf32_bits(St[(k0 + t4) * SP + 8 * nt + g8]),
                                            tf32_bits(St[(k0 + t4 + 4) * SP + 8 * nt + g8])};
                    mma_tf32((ks & 1) ? acc2[nt] : acc[nt], a, bb);
                }
            }
        }
        cp_async_wait<0>();  // this block's K_tilde, U, O_intra, e^gamma
        __syncthreads();     // (1) [W; Qe] and S^T reads done everywhere
        if (b + 1 < nb) load_wq(b + 1);
        cp_async_commit();
        // U' (warps 0-3) and outputs (warps 4-7)
        {
            const int nrow = min(kBlock, s.n - b * kBlock);
            const int rbase = 16 * (warp & 3) + g8;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int c = 8 * nt + 2 * t4;
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int i = rbase + 8 * hh;
                    const float z0 = acc[nt][2 * hh] + acc2[nt][2 * hh];
                    const float z1 = acc[nt][2 * hh + 1] + acc2[nt][2 * hh + 1];
                    if (warp < 4) {
                        Ups[i * SP + c] = tf32_round(Us[i * DS + c] - z0);
                        Ups[i * SP + c + 1] = tf32_round(Us[i * DS + c + 1] - z1);
                    } else if (i < nrow) {
                        const float o0 = z0 + Ois[i * DS + c], o1 = z1 + Ois[i * DS + c + 1];
                        const int64_t oi = ((s.row0 + (int64_t)b * kBlock + i) * Hv + h) * D + c0 + c;
                        if (p.out_bf16) {
                            *reinterpret_cast<__nv_bfloat162 *>(static_cast<__nv_bfloat16 *>(p.out) + oi) =
                                __floats2bfloat162_rn(o0, o1);
                        } else {
                            *reinterpret_cast<float2 *>(static_cast<float *>(p.out) + oi) = make_float2(o0, o1);
                        }
                    }
                }
            }
        }
        __syncthreads();  // (2) U' complete
        // S^T <- e^{gamma_63} S^T + K_tilde^T U'   (D / 16 warps own the state rows)
        if (16 * warp < D) {
            const float e = egs[0];
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
#pragma unroll
            for (int ks = 0; ks < kBlock / 8; ++ks) {
                const int k0 = 8 * ks;
                const uint32_t a[4] = {__float_as_uint(Kts[(k0 + t4) * LK + m0]),
                                       __float_as_uint(Kts[(k0 + t4) * LK + m0 + 8]),
                                       __float_as_uint(Kts[(k0 + t4 + 4) * LK + m0]),
                                       __float_as_uint(Kts[(k0 + t4 + 4) * LK + m0 + 8])};
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
        __syncthreads();  // (3) K_tilde, U, O_intra, e^gamma consumed; S^T updated
        if (b + 1 < nb) load_rest(b + 1);
        cp_async_commit();
        cp_async_wait<1>();  // next [W; Qe] landed (the rest may still be in flight)
        __syncthreads();     // (4)
    }
    cp_async_wait<0>();
    __syncthreads();
    for (int e = t; e < D * DS; e += kThreads) Sg[(int64_t)(e / DS) * D + c0 + e % DS] = St[(e / DS) * SP + e % DS];
}

template <int D, int DS>
static cudaError_t launch(const LaunchCommon &p, cudaStream_t st) {
    constexpr int LW = D + 4, LK = D + 8, SP = DS == 8 ? 8 : DS + 8;
    constexpr size_t smem =
        sizeof(float) * (2 * kBlock * LW + kBlock * LK + D * SP + kBlock * SP + 2 * kBlock * DS + 4);
    auto k = chain_tc_kernel<D, DS>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    k<<<p.n_sess * p.Hv * (D / DS), kThreads, smem, st>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn

cudaError_t gdn_launch_chain_tc(const gdn::LaunchCommon &p, int D, cudaStream_t st) {
    return D == 64 ? gdn::launch<64, 16>(p, st) : gdn::launch<128, 16>(p, st);
}
