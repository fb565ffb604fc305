// Conv-state commit, state copy (checkpoint capture / restore, session zeroing)
// and the one-token decode step.
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

// Two independent 16-byte-vector copies in one launch; a null source zero-fills.
__global__ void __launch_bounds__(256) copy2_kernel(uint4 *d0, const uint4 *s0, size_t n0, uint4 *d1,
                                                    const uint4 *s1, size_t n1) {
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n0 + n1; i += stride) {
        if (i < n0) d0[i] = s0 ? s0[i] : make_uint4(0, 0, 0, 0);
        else d1[i - n0] = s1 ? s1[i - n0] : make_uint4(0, 0, 0, 0);
    }
}

// Sum over the 32 lanes of a warp of 16 per-lane values, scattered: afterwards
// lanes 2c and 2c + 1 both hold the warp's total of value c (16 shuffles in all).
__device__ __forceinline__ float warp_reduce_scatter16(float (&v)[16]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16, half = 8; o >= 2; o >>= 1, half >>= 1) {
        const bool up = lane & o;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = up ? v[i] : v[i + half];
            const float keep = up ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 1);
}

// One token of one session: CTA (session, 16-column slice of d_v) x v-head, thread i owns row i of the
// slice of S^T (d_k x 16, in registers).
//   u = beta (v - alpha S k),  S^T <- alpha S^T + k u^T,  o = S q
// (the gated delta rule step with alpha = exp(g)); the conv state is committed by conv_commit_kernel.
template <int D, typename InT>
__global__ void __launch_bounds__(D) decode_kernel(const LaunchCommon p, int64_t ch) {
    constexpr int SC = 16, NW = D / 32, NSL = D / SC;
    __shared__ float red[2][NW], part[NW][SC], vsh[SC], ush[SC];
    const int si = blockIdx.x / NSL, sl = blockIdx.x % NSL, c0 = sl * SC;
    const SessRef s = p.s[si];
    const int h = blockIdx.y, hk = h / p.G, t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int64_t nq = (int64_t)p.Hk * D, nv = (int64_t)p.Hv * D;
    const InT *cw = static_cast<const InT *>(p.conv_w);
    const InT *cs = static_cast<const InT *>(s.conv);
    auto conv1 = [&](const void *xp, int64_t ld, int64_t col, int64_t chan) {
        float w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) w[i] = to_f(cw[chan * 4 + i]);
        const float x0 = to_f(static_cast<const InT *>(xp)[s.row0 * ld + col]);
        return conv_tap<InT>(w, to_f(cs[chan]), to_f(cs[ch + chan]), to_f(cs[2 * ch + chan]), x0, p.act);
    };
    // the slice of S^T: row t, columns c0 .. c0 + 15
    float *Srow = s.S + (int64_t)h * D * D + (int64_t)t * D + c0;
    float st[SC];
#pragma unroll
    for (int c = 0; c < SC; c += 4) {
        const float4 v = *reinterpret_cast<const float4 *>(Srow + c);
        st[c] = v.x; st[c + 1] = v.y; st[c + 2] = v.z; st[c + 3] = v.w;
    }
    const float yq = conv1(p.xq, nq, (int64_t)hk * D + t, (int64_t)hk * D + t);
    const float yk = conv1(p.xk, nq, (int64_t)hk * D + t, nq + (int64_t)hk * D + t);
    if (t < SC) vsh[t] = conv1(p.xv, nv, (int64_t)h * D + c0 + t, 2 * nq + (int64_t)h * D + c0 + t);
    float sq = yq * yq, sk = yk * yk;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
    }
    if (lane == 0) { red[0][warp] = sq; red[1][warp] = sk; }
    __syncthreads();
    float tq = 0.f, tk = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) { tq += red[0][w]; tk += red[1][w]; }
    const float qt = yq * (p.q_scale / sqrtf(tq + p.eps));
    const float kt = yk * (1.f / sqrtf(tk + p.eps));
    const float alpha = expf(p.g[s.row0 * p.Hv + h]), b = p.beta[s.row0 * p.Hv + h];

    // (S k)_j over the slice's columns: column sums of k_t S[t][j]
    float v[SC];
#pragma unroll
    for (int c = 0; c < SC; ++c) v[c] = kt * st[c];
    float r = warp_reduce_scatter16(v);
    if (!(lane & 1)) part[warp][lane >> 1] = r;
    __syncthreads();
    if (t < SC) {
        float kS = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) kS += part[w][t];
        ush[t] = b * (vsh[t] - alpha * kS);
    }
    __syncthreads();
    // S^T <- alpha S^T + k u^T, written back; o_j = (S q)_j
#pragma unroll
    for (int c = 0; c < SC; ++c) {
        st[c] = fmaf(kt, ush[c], alpha * st[c]);
        v[c] = st[c] * qt;
    }
#pragma unroll
    for (int c = 0; c < SC; c += 4) *reinterpret_cast<float4 *>(Srow + c) = make_float4(st[c], st[c + 1], st[c + 2], st[c + 3]);
    r = warp_reduce_scatter16(v);
    if (!(lane & 1)) part[warp][lane >> 1] = r;   // the (S k) partials were consumed before the barrier above
    __syncthreads();
    if (t < SC) {
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) o += part[w][t];
        const int64_t oi = (s.row0 * p.Hv + h) * D + c0 + t;
        if (p.out_bf16) static_cast<__nv_bfloat16 *>(p.out)[oi] = __float2bfloat16_rn(o);
        else static_cast<float *>(p.out)[oi] = o;
    }
}

}  // namespace gdn

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
    gdn::copy2_kernel<<<blocks, 256, 0, st>>>(static_cast<uint4 *>(dst0), static_cast<const uint4 *>(src0),
                                              bytes0 / 16, static_cast<uint4 *>(dst1),
                                              static_cast<const uint4 *>(src1), bytes1 / 16);
    return cudaGetLastError();
}

cudaError_t gdn_launch_decode(const gdn::LaunchCommon &p, int D, int in_bf16, int64_t ch, cudaStream_t st) {
    using namespace gdn;
    dim3 grid(p.n_sess * (D / 16), p.Hv);
    if (D == 64) {
        if (in_bf16) decode_kernel<64, __nv_bfloat16><<<grid, 64, 0, st>>>(p, ch);
        else decode_kernel<64, float><<<grid, 64, 0, st>>>(p, ch);
    } else {
        if (in_bf16) decode_kernel<128, __nv_bfloat16><<<grid, 128, 0, st>>>(p, ch);
        else decode_kernel<128, float><<<grid, 128, 0, st>>>(p, ch);
    }
    return cudaGetLastError();
}
