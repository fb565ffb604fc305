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
    const InT old[3] = {cs[chan], cs[ch + chan], cs[2 * ch + chan]};
    InT nw[3];
#pragma unroll
    for (int r = 0; r < 3; ++r) {
        const int pos = s.n - 3 + r;
        nw[r] = pos >= 0 ? x[(s.row0 + pos) * ld + col] : old[3 + pos];
    }
#pragma unroll
    for (int r = 0; r < 3; ++r) cs[r * ch + chan] = nw[r];
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

// One token of one session and v-head; thread j owns column j of S^T.
//   u = beta (v - alpha S k),  S^T <- alpha S^T + k u^T,  o = S q
// (the gated delta rule step with alpha = exp(g)).
template <int D, typename InT>
__global__ void __launch_bounds__(D) decode_kernel(const LaunchCommon p, int64_t ch) {
    __shared__ float qs[D], ks[D], red[2][D / 32];
    const SessRef s = p.s[blockIdx.x];
    const int h = blockIdx.y, hk = h / p.G, t = threadIdx.x;
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
    const float yq = conv1(p.xq, nq, (int64_t)hk * D + t, (int64_t)hk * D + t);
    const float yk = conv1(p.xk, nq, (int64_t)hk * D + t, nq + (int64_t)hk * D + t);
    const float yv = conv1(p.xv, nv, (int64_t)h * D + t, 2 * nq + (int64_t)h * D + t);
    float sq = yq * yq, sk = yk * yk;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
    }
    if ((t & 31) == 0) { red[0][t >> 5] = sq; red[1][t >> 5] = sk; }
    __syncthreads();
    float tq = 0.f, tk = 0.f;
#pragma unroll
    for (int w = 0; w < D / 32; ++w) { tq += red[0][w]; tk += red[1][w]; }
    qs[t] = yq * (p.q_scale / sqrtf(tq + p.eps));
    ks[t] = yk * (1.f / sqrtf(tk + p.eps));
    __syncthreads();

    float *S = s.S + (int64_t)h * D * D;
    const float alpha = expf(p.g[s.row0 * p.Hv + h]), b = p.beta[s.row0 * p.Hv + h];
    float kS = 0.f;
    for (int i = 0; i < D; ++i) kS = fmaf(ks[i], S[i * D + t], kS);
    const float u = b * (yv - alpha * kS);
    float o = 0.f;
    for (int i = 0; i < D; ++i) {
        const float sn = fmaf(ks[i], u, alpha * S[i * D + t]);
        S[i * D + t] = sn;
        o = fmaf(sn, qs[i], o);
    }
    const int64_t oi = (s.row0 * p.Hv + h) * D + t;
    if (p.out_bf16) static_cast<__nv_bfloat16 *>(p.out)[oi] = __float2bfloat16_rn(o);
    else static_cast<float *>(p.out)[oi] = o;
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
    dim3 grid(p.n_sess, p.Hv);
    if (D == 64) {
        if (in_bf16) decode_kernel<64, __nv_bfloat16><<<grid, 64, 0, st>>>(p, ch);
        else decode_kernel<64, float><<<grid, 64, 0, st>>>(p, ch);
    } else {
        if (in_bf16) decode_kernel<128, __nv_bfloat16><<<grid, 128, 0, st>>>(p, ch);
        else decode_kernel<128, float><<<grid, 128, 0, st>>>(p, ch);
    }
    return cudaGetLastError();
}
