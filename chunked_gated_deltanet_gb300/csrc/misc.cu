// Conv-state commit, state copy (checkpoint capture / restore, session zeroing)
// and the one-token decode step (which commits its own conv state).
#include <algorithm>

#include "common.cuh"

namespace gdn {

// New conv state of each session: the raw inputs at its last three processed
// positions (taken from the packed inputs, or shifted from the old state when
// fewer than three tokens were processed). Bitwise copies of input values.
template <typename InT>
__global__ void __launch_bounds__(256) conv_commit_kernel(const LaunchCommon p, int D, int64_t ch) {
    const SessRef s = p.s[blockIdx.y];
    const int64_t chan = (int64_t)blockIdx.x * 256 + threadIdx.x;
    if (chan >= ch || s.n <= 0) return;
    const int64_t nq = (int64_t)p.Hk * D, nv = (int64_t)p.Hv * D;
    const InT *x;
    int64_t col, ld;
    if (chan < nq) { x = static_cast<const InT *>(p.xq); col = chan; ld = nq; }
    else if (chan < 2 * nq) { x = static_cast<const InT *>(p.xk); col = chan - nq; ld = nq; }
    else { x = static_cast<const InT *>(p.xv); col = chan - 2 * nq; ld = nv; }
    InT *cs = static_cast<InT *>(s.conv);
    const InT *cs0 = static_cast<const InT *>(s.conv0);
    const InT o0 = cs0[chan], o1 = cs0[ch + chan], o2 = cs0[2 * ch + chan];
    InT nw[3];
#pragma unroll
    for (int r = 0; r < 3; ++r) {
        const int pos = s.n - 3 + r;
        nw[r] = pos >= 0 ? x[(s.row0 + pos) * ld + col] : (pos == -3 ? o0 : (pos == -2 ? o1 : o2));
    }
#pragma unroll
    for (int r = 0; r < 3; ++r) cs[r * ch + chan] = nw[r];
    if (s.conv_cap) {
        InT *cc = static_cast<InT *>(s.conv_cap);
#pragma unroll
        for (int r = 0; r < 3; ++r) cc[r * ch + chan] = nw[r];
    }
}

// Two independent 16-byte-vector copies in one launch; a null source zero-fills. Launched with
// programmatic stream serialization: it waits for earlier work before touching memory, then lets the next
// kernel start as its CTAs leave.
__global__ void __launch_bounds__(256) copy2_kernel(uint4 *d0, const uint4 *s0, size_t n0, uint4 *d1,
                                                    const uint4 *s1, size_t n1) {
    grid_dep_wait();
    grid_dep_launch();
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n0 + n1; i += stride) {
        if (i < n0) d0[i] = s0 ? s0[i] : make_uint4(0, 0, 0, 0);
        else d1[i - n0] = s1 ? s1[i - n0] : make_uint4(0, 0, 0, 0);
    }
}

// One token of one session for one q/k head and its G v-heads: CTA (session, q/k head), 256 threads.
// Thread t owns columns 4 (t % (D/4)) .. + 3 of rows t / (D/4) + NRG i of S^T (NRG = 1024 / D row
// groups), so every warp-wide access of the state reads or writes whole rows in 16-byte vectors.
//   u = beta (v - alpha S k),  S^T <- alpha S^T + k u^T,  o = S q
// (the gated delta rule step with alpha = exp(g)). Sums over d_k go in a fixed order: each thread over
// its rows in increasing order, then the row groups in increasing order, so a session's result does not
// depend on the batch. The CTA is the only reader of its channels' conv state (q and k of its head, v of
// its v-heads), and each channel's old state is read by the one thread that writes its new state, so
// the conv state is committed in place without a separate launch.
// A call of more than 64 sessions is several launches (chunks) over disjoint sessions, each letting the next
// start as its CTAs leave: chunk 0 waits for earlier work before it lets the next one launch, so every
// chunk starts after that work; a later chunk waits for the chunk before it only at its end, so that the
// last chunk completes after every other one and work after the call waits for the whole step.
template <int D, typename InT>
__global__ void __launch_bounds__(256) decode_kernel(const LaunchCommon p, int64_t ch, int chunk) {
    if (chunk == 0) grid_dep_wait();   // inputs, states and conv states, written by earlier work
    grid_dep_launch();
    constexpr int NT = 256, LPR = D / 4, NRG = NT / LPR, RPT = D / NRG, NW = NT / 32;
    static_assert(2 * D <= NT && RPT * NRG == D, "thread map");
    __shared__ float qk[2][D], vv[D], uu[D], red[NRG][D], ss[NW];
    const SessRef s = p.s[blockIdx.x];
    const int hk = blockIdx.y, t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int c0 = 4 * (t % LPR), rg = t / LPR;
    const int64_t nq = (int64_t)p.Hk * D, nv = (int64_t)p.Hv * D;
    const InT *cw = static_cast<const InT *>(p.conv_w);
    const InT *cs0 = static_cast<const InT *>(s.conv0);
    InT *cs = static_cast<InT *>(s.conv);
    // conv of one channel from its raw input x0 and old state, and the channel's new state [old1, old2, x0]
    auto conv1 = [&](InT x0, int64_t chan) {
        float w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = to_f(cw[chan * 4 + i]);
        const InT o0 = cs0[chan], o1 = cs0[ch + chan], o2 = cs0[2 * ch + chan];
        const float y = conv_tap<InT>(w, to_f(o0), to_f(o1), to_f(o2), to_f(x0), p.act);
        cs[chan] = o1;
        cs[ch + chan] = o2;
        cs[2 * ch + chan] = x0;
        return y;
    };
    auto load_state = [&](float4 (&st)[RPT], int h) {
        const float *S0 = s.S0 + (int64_t)h * D * D;
#pragma unroll
        for (int i = 0; i < RPT; ++i) st[i] = *reinterpret_cast<const float4 *>(S0 + (int64_t)(rg + NRG * i) * D + c0);
    };
    float4 st[RPT];
    load_state(st, hk * p.G);   // in flight during the conv of q and k

    // q (threads 0..D-1) and k (threads D..2D-1), L2-normalised into qk
    if (t < 2 * D) {
        const int c = t % D;
        const bool isk = t >= D;
        const InT *x = static_cast<const InT *>(isk ? p.xk : p.xq);
        const float y = conv1(x[s.row0 * nq + (int64_t)hk * D + c], (isk ? nq : 0) + (int64_t)hk * D + c);
        float sq = y * y;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
        if (lane == 0) ss[warp] = sq;
        qk[isk][c] = y;
    }
    __syncthreads();
    if (t < 2 * D) {
        const int c = t % D, w0 = t < D ? 0 : D / 32;
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < D / 32; ++w) tot += ss[w0 + w];
        qk[t >= D][c] *= (t < D ? p.q_scale : 1.f) / sqrtf(tot + p.eps);
    }

    for (int gi = 0; gi < p.G; ++gi) {
        const int h = hk * p.G + gi;
        if (gi > 0) load_state(st, h);
        if (t < D) vv[t] = conv1(static_cast<const InT *>(p.xv)[s.row0 * nv + (int64_t)h * D + t], 2 * nq + (int64_t)h * D + t);
        const float alpha = expf(p.g[s.row0 * p.Hv + h]), b = p.beta[s.row0 * p.Hv + h];
        __syncthreads();   // q, k, v of this head are in shared memory; red and uu are free

        // (S k) over this thread's rows, then over the row groups
        float4 pk = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            const float kr = qk[1][rg + NRG * i];
            pk.x = fmaf(kr, st[i].x, pk.x); pk.y = fmaf(kr, st[i].y, pk.y);
            pk.z = fmaf(kr, st[i].z, pk.z); pk.w = fmaf(kr, st[i].w, pk.w);
        }
        *reinterpret_cast<float4 *>(&red[rg][c0]) = pk;
        __syncthreads();
        if (t < D) {
            float kS = 0.f;
#pragma unroll
            for (int r = 0; r < NRG; ++r) kS += red[r][t];
            uu[t] = b * (vv[t] - alpha * kS);
        }
        __syncthreads();
        // S^T <- alpha S^T + k u^T, written back; o = S q over this thread's rows, then the row groups
        const float4 u = *reinterpret_cast<const float4 *>(&uu[c0]);
        float *Sh = s.S + (int64_t)h * D * D;
        float4 po = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < RPT; ++i) {
            const int r = rg + NRG * i;
            const float kr = qk[1][r], qr = qk[0][r];
            float4 v = st[i];
            v.x = fmaf(kr, u.x, alpha * v.x); v.y = fmaf(kr, u.y, alpha * v.y);
            v.z = fmaf(kr, u.z, alpha * v.z); v.w = fmaf(kr, u.w, alpha * v.w);
            *reinterpret_cast<float4 *>(Sh + (int64_t)r * D + c0) = v;
            po.x = fmaf(qr, v.x, po.x); po.y = fmaf(qr, v.y, po.y);
            po.z = fmaf(qr, v.z, po.z); po.w = fmaf(qr, v.w, po.w);
        }
        *reinterpret_cast<float4 *>(&red[rg][c0]) = po;   // every read of the (S k) partials preceded the barrier above
        __syncthreads();
        if (t < D) {
            float o = 0.f;
#pragma unroll
            for (int r = 0; r < NRG; ++r) o += red[r][t];
            const int64_t oi = (s.row0 * p.Hv + h) * D + t;
            if (p.out_bf16) static_cast<__nv_bfloat16 *>(p.out)[oi] = __float2bfloat16_rn(o);
            else static_cast<float *>(p.out)[oi] = o;
        }
        __syncthreads();   // red, vv and uu are read before the next head writes them
    }
    if (chunk > 0) grid_dep_wait();   // the chunk before this one is complete
}

// g and beta from raw per-token projections (the raw-gate variant, the usual Gated-DeltaNet
// parametrisation; the pages take g and beta as given):
//   g = -exp(A_log[h]) * softplus(a + dt_bias[h]),  beta = 1 / (1 + exp(-b)),
// softplus(x) = max(x, 0) + log1p(exp(-|x|)), element i of [tokens][Hv] belonging to head i % Hv.
__global__ void __launch_bounds__(256) gates_kernel(const float *a, const float *b, const float *A_log,
                                                    const float *dt_bias, int64_t n, int Hv, float *g, float *beta) {
    for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (int64_t)gridDim.x * 256) {
        const int h = (int)(i % Hv);
        const float x = a[i] + dt_bias[h];
        const float sp = fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
        g[i] = -expf(A_log[h]) * sp;
        beta[i] = 1.f / (1.f + expf(-b[i]));
    }
}

}  // namespace gdn

cudaError_t gdn_launch_gates(const float *a, const float *b, const float *A_log, const float *dt_bias, int64_t n,
                             int Hv, float *g, float *beta, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    const int64_t blocks = std::min<int64_t>((n + 255) / 256, 152 * 8);
    gdn::gates_kernel<<<(unsigned)blocks, 256, 0, st>>>(a, b, A_log, dt_bias, n, Hv, g, beta);
    return cudaGetLastError();
}

cudaError_t gdn_launch_conv_commit(const gdn::LaunchCommon &p, int D, int in_bf16, int64_t ch, cudaStream_t st) {
    using namespace gdn;
    dim3 grid((unsigned)((ch + 255) / 256), p.n_sess);
    if (in_bf16) conv_commit_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>(p, D, ch);
    else conv_commit_kernel<float><<<grid, 256, 0, st>>>(p, D, ch);
    return cudaGetLastError();
}

cudaError_t gdn_launch_copy(void *dst0, const void *src0, size_t bytes0, void *dst1, const void *src1,
                            size_t bytes1, cudaStream_t st) {
    const size_t n = (bytes0 + bytes1) / 16;
    if (n == 0) return cudaSuccess;
    unsigned blocks = (unsigned)((n + 255) / 256);
    if (blocks > 152u * 8u) blocks = 152u * 8u;
    const cudaError_t e = gdn_launch_pdl(gdn::copy2_kernel, blocks, 256, 0, st, static_cast<uint4 *>(dst0),
                                         static_cast<const uint4 *>(src0), bytes0 / 16, static_cast<uint4 *>(dst1),
                                         static_cast<const uint4 *>(src1), bytes1 / 16);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t gdn_launch_decode(const gdn::LaunchCommon &p, int D, int in_bf16, int64_t ch, int chunk, cudaStream_t st) {
    using namespace gdn;
    const dim3 grid(p.n_sess, p.Hk);
    cudaError_t e;
    if (D == 64)
        e = in_bf16 ? gdn_launch_pdl(decode_kernel<64, __nv_bfloat16>, grid, 256, 0, st, p, ch, chunk)
                    : gdn_launch_pdl(decode_kernel<64, float>, grid, 256, 0, st, p, ch, chunk);
    else
        e = in_bf16 ? gdn_launch_pdl(decode_kernel<128, __nv_bfloat16>, grid, 256, 0, st, p, ch, chunk)
                    : gdn_launch_pdl(decode_kernel<128, float>, grid, 256, 0, st, p, ch, chunk);
    return e != cudaSuccess ? e : cudaGetLastError();
}
