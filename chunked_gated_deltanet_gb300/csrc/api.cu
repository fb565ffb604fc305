// C ABI of the library (declared in include/gdn.h): argument validation on the
// host before any device work, workspace layout, and launch orchestration.
#include "gdn.h"
#include "common.cuh"
#include "host.h"

#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <random>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <vector>

#define GDN_API extern "C" __attribute__((visibility("default")))

using gdn::kBlock;
using gdn::LaunchCommon;

namespace gdn_host {

thread_local char g_err[512] = "";

gdn_status fail(gdn_status st, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return st;
}

gdn_status cuda_fail(cudaError_t e, const char *what) {
    return fail(GDN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t channels(const gdn_layer_desc *d) {
    return 2LL * d->n_qk_heads * d->d_k + (int64_t)d->n_v_heads * d->d_v;
}

size_t in_elt(const gdn_layer_desc *d) { return d->in_dtype == GDN_BF16 ? 2 : 4; }

gdn_status check_desc(const gdn_layer_desc *d) {
    if (!d) return fail(GDN_ERR_INVALID_ARG, "layer description is NULL");
    if (d->n_qk_heads < 1 || d->n_v_heads < 1 || d->n_v_heads % d->n_qk_heads != 0 || d->n_v_heads > 65535)
        return fail(GDN_ERR_SHAPE, "heads: need 1 <= Hk, Hv a multiple of Hk, Hv <= 65535 (Hk=%d, Hv=%d)",
                    d->n_qk_heads, d->n_v_heads);
    if ((d->d_k != 64 && d->d_k != 128) || d->d_v != d->d_k)
        return fail(GDN_ERR_SHAPE, "head dims: need d_k = d_v in {64, 128} (d_k=%d, d_v=%d)", d->d_k, d->d_v);
    if (d->grid_c < 64 || d->grid_c > 4096 || d->grid_c % 64 != 0)
        return fail(GDN_ERR_SHAPE, "grid_c must be a multiple of 64 in [64, 4096] (got %d)", d->grid_c);
    if (d->in_dtype != GDN_BF16 && d->in_dtype != GDN_FP32)
        return fail(GDN_ERR_SHAPE, "in_dtype must be GDN_BF16 or GDN_FP32 (got %d)", d->in_dtype);
    if (d->out_dtype != GDN_BF16 && d->out_dtype != GDN_FP32)
        return fail(GDN_ERR_SHAPE, "out_dtype must be GDN_BF16 or GDN_FP32 (got %d)", d->out_dtype);
    if (d->conv_act != GDN_CONV_NONE && d->conv_act != GDN_CONV_SILU)
        return fail(GDN_ERR_SHAPE, "conv_act must be GDN_CONV_NONE or GDN_CONV_SILU (got %d)", d->conv_act);
    if (!(d->l2_eps > 0.f) || !std::isfinite(d->l2_eps) || !std::isfinite(d->q_scale))
        return fail(GDN_ERR_INVALID_ARG, "l2_eps must be finite and > 0, q_scale finite");
    return GDN_OK;
}

uint64_t tag_of(const gdn_layer_desc *d) {
    // FNV-1a over a format version and every field of the description
    uint64_t h = 1469598103934665603ULL;
    auto mix = [&](uint32_t v) {
        for (int i = 0; i < 4; ++i) { h ^= (v >> (8 * i)) & 0xffu; h *= 1099511628211ULL; }
    };
    mix(0x31444447u);  // "GDD1": state layout version
    const int32_t f[8] = {d->n_qk_heads, d->n_v_heads, d->d_k, d->d_v, d->grid_c, d->in_dtype, d->out_dtype, d->conv_act};
    for (int32_t v : f) mix((uint32_t)v);
    uint32_t b;
    std::memcpy(&b, &d->q_scale, 4); mix(b);
    std::memcpy(&b, &d->l2_eps, 4); mix(b);
    return h ? h : 1;
}

gdn_status check_state(const gdn_layer_desc *d, const gdn_session *s, const char *what, bool need_present) {
    if (!s) return fail(GDN_ERR_INVALID_ARG, "%s is NULL", what);
    if (!s->S || !s->conv || !aligned16(s->S) || !aligned16(s->conv))
        return fail(GDN_ERR_INVALID_ARG, "%s: S and conv must be non-NULL and 16-byte aligned", what);
    if (s->tag != tag_of(d))
        return fail(GDN_ERR_STATE_MISMATCH, "%s belongs to another layer description (tag %llx, expected %llx)",
                    what, (unsigned long long)s->tag, (unsigned long long)tag_of(d));
    if (need_present && s->committed < 0)
        return fail(GDN_ERR_STATE_MISMATCH, "%s is a missing slot (committed = %lld)", what, (long long)s->committed);
    return GDN_OK;
}

}  // namespace gdn_host

using namespace gdn_host;

namespace {

// Workspace layout for a launch of up to nblk blocks. Offsets count from the workspace pointer
// rounded up to 256 bytes (the kernels' widest stores want 32-byte alignment); `bytes` includes
// that slack.
struct WsLayout {
    size_t qk_off, wu_off, flags_off, bytes;
};
constexpr size_t kWsAlign = 256;
char *ws_base(void *workspace) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(workspace);
    return reinterpret_cast<char *>((a + kWsAlign - 1) & ~(uintptr_t)(kWsAlign - 1));
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

WsLayout ws_layout(const gdn_layer_desc *d, int64_t nblk) {
    WsLayout L;
    const int D = d->d_k;
    L.flags_off = 0;
    if (d->in_dtype == GDN_BF16) {  // tensor-core path: one record per (block, v-head)
        L.qk_off = 0;
        L.wu_off = 0;
        const size_t rec = D == 128 ? gdn::rec16::kBytes : gdn::rec_floats(D) * sizeof(float);
        L.flags_off = align256((size_t)nblk * d->n_v_heads * rec);
        // d = 128: a 64-bit publication flag per (block, q/k head) for the one-launch prefill
        const size_t flags = D == 128 ? align256((size_t)nblk * d->n_qk_heads * sizeof(unsigned long long)) : 0;
        L.bytes = kWsAlign + L.flags_off + flags;
        return L;
    }
    L.qk_off = 0;
    L.wu_off = align256((size_t)nblk * d->n_qk_heads * gdn::qk_floats(D) * sizeof(float));
    L.bytes = kWsAlign + L.wu_off + align256((size_t)nblk * d->n_v_heads * gdn::wu_floats(D) * sizeof(float));
    return L;
}

// Epochs of the one-launch prefill's publication flags: a fresh value per launch, starting from a random
// 64-bit base, so that a flag left by an earlier call (or whatever a fresh workspace holds) does not read as
// published except by a 2^-64 coincidence.
std::atomic<unsigned long long> g_epoch{[] {
    std::random_device rd;
    return ((unsigned long long)rd() << 32) ^ (unsigned long long)rd() ^ 0x9e3779b97f4a7c15ULL;
}()};

// Bounded waits: default poll limit, and the test hook that makes the next launches' waits run out.
constexpr long long kDefaultWaitLimit = 1LL << 24;
long long g_wait_limit = kDefaultWaitLimit;
int g_skip_first_copy = 0;

void fill_common(LaunchCommon &p, const gdn_layer_desc *d, const void *xq, const void *xk, const void *xv,
                 const float *g, const float *beta, const void *conv_w, void *out) {
    std::memset(&p, 0, sizeof(p));
    for (int i = 0; i < gdn::kLaunchSessions; ++i) p.order[i] = (unsigned char)i;
    p.wait_limit = g_wait_limit;
    p.debug_skip_first_copy = g_skip_first_copy;
    p.blk_lo = 0;
    p.xq = xq; p.xk = xk; p.xv = xv; p.g = g; p.beta = beta; p.conv_w = conv_w; p.out = out;
    p.Hk = d->n_qk_heads; p.Hv = d->n_v_heads; p.G = d->n_v_heads / d->n_qk_heads;
    p.act = d->conv_act; p.out_bf16 = d->out_dtype == GDN_BF16;
    p.q_scale = d->q_scale; p.eps = d->l2_eps;
}

// 2-D tensor map over a row-major bf16 [rows][cols] input, boxes of 64 rows x 128 channels.
// cuTensorMapEncodeTiled is reached through the runtime's driver entry point (no libcuda link).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

cudaError_t encode_rows_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols) {
    const auto fn = tensor_map_encoder();
    if (!fn) return cudaErrorNotSupported;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)std::max<int64_t>(rows, 1)};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {128, (cuuint32_t)kBlock};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// ---- optional per-kernel event timing ----
enum Kind { K_PREP = 0, K_CONV = 1, K_STATE = 2, K_COPY = 3, K_DECODE = 4, K_GATES = 5, K_PREP_TAIL = 6, K_FUSED = 7,
            K_KINDS = 8 };
const char *const kKindName[K_KINDS] = {"prep_wy", "conv_commit", "state_output", "state_copy", "decode", "gates",
                                        "prep_wy_tail", "prefill_fused"};

struct Timing {
    bool on = false;
    int cap = 0, used = 0;
    std::vector<cudaEvent_t> ev;  // 2 per timed launch
    std::vector<int> kind;
    int64_t launches[K_KINDS] = {};
};
Timing g_timing;

template <class F>
cudaError_t launch_k(Kind k, cudaStream_t st, F &&f) {
    Timing &T = g_timing;
    if (!T.on) return f();
    T.launches[k]++;
    if (T.used >= T.cap) return f();
    cudaEvent_t a = T.ev[2 * T.used], b = T.ev[2 * T.used + 1];
    cudaError_t e = cudaEventRecord(a, st);
    if (e != cudaSuccess) return e;
    e = f();
    if (e != cudaSuccess) return e;
    e = cudaEventRecord(b, st);
    if (e == cudaSuccess) T.kind[T.used++] = k;
    return e;
}

}  // namespace

GDN_API gdn_status gdn_timing_begin(int32_t max_launches) {
    Timing &T = g_timing;
    if (T.on) return fail(GDN_ERR_INVALID_ARG, "timing already recording");
    if (max_launches < 0 || max_launches > (1 << 22)) return fail(GDN_ERR_INVALID_ARG, "max_launches out of range");
    for (cudaEvent_t e : T.ev) cudaEventDestroy(e);
    T.ev.assign(2 * (size_t)max_launches, nullptr);
    for (auto &e : T.ev) {
        cudaError_t r = cudaEventCreate(&e);
        if (r != cudaSuccess) return cuda_fail(r, "event creation");
    }
    T.kind.assign(max_launches, 0);
    T.cap = max_launches;
    T.used = 0;
    for (auto &l : T.launches) l = 0;
    T.on = true;
    return GDN_OK;
}

GDN_API gdn_status gdn_timing_end(gdn_kernel_time *out, int32_t max_kinds, int32_t *n_kinds) {
    Timing &T = g_timing;
    if (!T.on) return fail(GDN_ERR_INVALID_ARG, "timing is not recording");
    T.on = false;
    double ms[K_KINDS] = {};
    int64_t timed[K_KINDS] = {};
    for (int i = 0; i < T.used; ++i) {
        cudaError_t r = cudaEventSynchronize(T.ev[2 * i + 1]);
        if (r != cudaSuccess) return cuda_fail(r, "event wait");
        float m = 0.f;
        r = cudaEventElapsedTime(&m, T.ev[2 * i], T.ev[2 * i + 1]);
        if (r != cudaSuccess) return cuda_fail(r, "event elapsed time");
        ms[T.kind[i]] += m;
        timed[T.kind[i]]++;
    }
    int n = 0;
    for (int k = 0; k < K_KINDS; ++k) {
        if (T.launches[k] == 0) continue;
        if (out && n < max_kinds) {
            std::memset(&out[n], 0, sizeof(out[n]));
            snprintf(out[n].name, sizeof(out[n].name), "%s", kKindName[k]);
            out[n].launches = T.launches[k];
            out[n].timed = timed[k];
            out[n].total_ms = ms[k];
        }
        ++n;
    }
    if (n_kinds) *n_kinds = n;
    return GDN_OK;
}

void gdn_internal_set_error(const char *msg) { snprintf(g_err, sizeof(g_err), "%s", msg); }

GDN_API uint64_t gdn_desc_tag(const gdn_layer_desc *desc) {
    if (check_desc(desc) != GDN_OK) return 0;
    return tag_of(desc);
}

GDN_API gdn_status gdn_desc_check(const gdn_layer_desc *desc) { return check_desc(desc); }

GDN_API size_t gdn_state_bytes(const gdn_layer_desc *d) {
    if (check_desc(d) != GDN_OK) return 0;
    return (size_t)d->n_v_heads * d->d_k * d->d_v * sizeof(float);
}

GDN_API size_t gdn_conv_state_bytes(const gdn_layer_desc *d) {
    if (check_desc(d) != GDN_OK) return 0;
    return 3 * (size_t)channels(d) * in_elt(d);
}

GDN_API gdn_status gdn_session_init(const gdn_layer_desc *d, gdn_session *s, float *S, void *conv,
                                    gdn_stream_t stream) {
    gdn_status st = check_desc(d);
    if (st != GDN_OK) return st;
    if (!s) return fail(GDN_ERR_INVALID_ARG, "session is NULL");
    if (!S || !conv || !aligned16(S) || !aligned16(conv))
        return fail(GDN_ERR_INVALID_ARG, "S and conv must be non-NULL and 16-byte aligned");
    cudaError_t e = launch_k(K_COPY, (cudaStream_t)stream, [&] {
        return gdn_launch_copy(S, nullptr, gdn_state_bytes(d), conv, nullptr, gdn_conv_state_bytes(d),
                               (cudaStream_t)stream);
    });
    if (e != cudaSuccess) return cuda_fail(e, "session zeroing");
    s->S = S; s->conv = conv; s->committed = 0; s->tag = tag_of(d);
    return GDN_OK;
}

GDN_API size_t gdn_workspace_size(const gdn_layer_desc *d, int64_t max_tokens, int32_t max_sessions) {
    if (check_desc(d) != GDN_OK || max_tokens < 0 || max_sessions < 1) return 0;
    const int64_t per_launch = std::min<int64_t>(max_sessions, gdn::kLaunchSessions);
    const int64_t nblk = (max_tokens + kBlock - 1) / kBlock + per_launch;
    return ws_layout(d, nblk).bytes;
}

namespace {

// Prefill of n sessions; with `prefix`, every session starts from the prefix's state (read in place) and
// receives its own result, as if the prefix had been restored into it first.
// Where to split a one-session bf16 launch (d = 128) whose prologue would end with a partial round: blocks
// [0, split) take whole rounds of one CTA per SM, and the tasks of the rest run, on the SMs the state pass
// of the first part leaves (its chain CTAs hold one SM each), while that state pass runs. 0: no split (no
// partial round, no free SMs, or the rest would outlast the first state pass). The times are those
// measured on GB300 for this layer: about 12.5 us per round of prologue tasks (one q/k head of a 64-token
// block per SM) and, for the state pass, kStateStepUs per block plus kStateFixedUs per launch, which the
// second state pass adds.
constexpr double kPrologueRoundUs = 12.5, kStateStepUs = 0.6, kStateFixedUs = 4.0;
static int tail_split(const LaunchCommon &p, const gdn_layer_desc *d) {
    if (p.n_sess != 1 || p.G != 1) return 0;
    int sms = 0;
    if (gdn_sm_count(&sms) != cudaSuccess) return 0;
    const int Hk = p.Hk, nblk = p.nblk;
    const int nchain = d->n_v_heads * (d->d_v / gdn_chain_umma_cols(d->n_v_heads, sms));
    const int free_sms = sms - nchain;
    if (nchain > sms || free_sms < 8) return 0;
    const int64_t ntask = (int64_t)nblk * Hk, rounds = (ntask + sms - 1) / sms;
    if (rounds < 2 || ntask % sms == 0) return 0;
    const int split = (int)((rounds - 1) * sms / Hk);   // blocks in whole rounds
    if (split < 1 || split >= nblk) return 0;
    const int64_t rest = (int64_t)(nblk - split) * Hk, rest_rounds = (rest + free_sms - 1) / free_sms;
    const double t_rest = kPrologueRoundUs * (double)rest_rounds, t_first_state = kStateStepUs * split + kStateFixedUs;
    // a round saved against a second state pass's fixed cost
    return t_rest <= t_first_state && kPrologueRoundUs > kStateFixedUs ? split : 0;
}

gdn_status prefill_impl(const gdn_layer_desc *d, gdn_session *sessions, int32_t n_sessions, const int64_t *cu,
                        const void *xq, const void *xk, const void *xv, const float *g, const float *beta,
                        const void *conv_w, uint32_t flags, void *out, int64_t *n_consumed, void *workspace,
                        size_t workspace_bytes, gdn_stream_t stream, const gdn_session *prefix,
                        gdn_session *ckpt) {
    gdn_status st = check_desc(d);
    if (st != GDN_OK) return st;
    if (prefix && (st = check_state(d, prefix, "prefix", true)) != GDN_OK) return st;
    if (ckpt && n_sessions >= 1)
        for (int i = 0; i < n_sessions; ++i)
            if (!ckpt[i].S || !ckpt[i].conv || !aligned16(ckpt[i].S) || !aligned16(ckpt[i].conv))
                return fail(GDN_ERR_INVALID_ARG, "checkpoint slot %d: buffers must be non-NULL and 16-byte aligned", i);
    if (flags & ~GDN_ALLOW_PARTIAL) return fail(GDN_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
    if (n_sessions < 1 || n_sessions > GDN_MAX_SESSIONS)
        return fail(GDN_ERR_INVALID_ARG, "n_sessions must be in [1, %d] (got %d)", GDN_MAX_SESSIONS, n_sessions);
    if (!sessions || !cu || !n_consumed) return fail(GDN_ERR_INVALID_ARG, "sessions, cu_seqlens, n_consumed must be non-NULL");
    if (cu[0] != 0) return fail(GDN_ERR_INVALID_ARG, "cu_seqlens[0] must be 0 (got %lld)", (long long)cu[0]);
    const bool partial = flags & GDN_ALLOW_PARTIAL;
    const int C = d->grid_c;
    std::vector<int64_t> nproc(n_sessions);
    int64_t total = 0;
    for (int i = 0; i < n_sessions; ++i) {
        const int64_t len = cu[i + 1] - cu[i];
        if (len < 0) return fail(GDN_ERR_INVALID_ARG, "cu_seqlens must be non-decreasing (at %d)", i);
        if (len > (int64_t)1 << 30) return fail(GDN_ERR_INVALID_ARG, "session %d: more than 2^30 tokens in one call", i);
        char what[48];
        snprintf(what, sizeof(what), prefix ? "branch %d" : "session %d", i);
        if ((st = check_state(d, &sessions[i], what, !prefix)) != GDN_OK) return st;
        const int64_t base = prefix ? prefix->committed : sessions[i].committed;
        if (!partial && base % C != 0)
            return fail(GDN_ERR_OFF_GRID, "%s is off grid (committed %lld, grid %d): only a partial call, "
                        "a decode step or a restore may follow", prefix ? "the prefix" : what, (long long)base, C);
        nproc[i] = partial ? len : (len / C) * C;
        total += nproc[i];
    }
    {
        std::vector<const void *> ptrs(n_sessions);
        for (int i = 0; i < n_sessions; ++i) ptrs[i] = sessions[i].S;
        if (prefix) ptrs.push_back(prefix->S);
        if (ckpt)
            for (int i = 0; i < n_sessions; ++i) ptrs.push_back(ckpt[i].S);
        std::sort(ptrs.begin(), ptrs.end());
        if (std::adjacent_find(ptrs.begin(), ptrs.end()) != ptrs.end())
            return fail(GDN_ERR_INVALID_ARG, prefix ? "the branches, the prefix and the checkpoints must be distinct"
                                                    : "the sessions and checkpoints of one call must be distinct");
    }
    // blocks per launch batch, and the workspace that needs
    int64_t max_batch_blocks = 0;
    for (int i0 = 0; i0 < n_sessions;) {
        int64_t nb = 0;
        int cnt = 0, i = i0;
        for (; i < n_sessions && cnt < gdn::kLaunchSessions; ++i)
            if (nproc[i] > 0) { nb += (nproc[i] + kBlock - 1) / kBlock; ++cnt; }
        max_batch_blocks = std::max(max_batch_blocks, nb);
        i0 = i;
    }
    if (total > 0) {
        if (!xq || !xk || !xv || !g || !beta || !conv_w || !out)
            return fail(GDN_ERR_INVALID_ARG, "input / output pointers must be non-NULL");
        if (!aligned16(xq) || !aligned16(xk) || !aligned16(xv) || !aligned16(conv_w) || !aligned16(out) ||
            (reinterpret_cast<uintptr_t>(g) & 3) || (reinterpret_cast<uintptr_t>(beta) & 3))
            return fail(GDN_ERR_INVALID_ARG, "xq, xk, xv, conv_w, out must be 16-byte aligned; g, beta 4-byte aligned");
        const WsLayout L = ws_layout(d, max_batch_blocks);
        if (!workspace || !aligned16(workspace) || workspace_bytes < L.bytes)
            return fail(GDN_ERR_WORKSPACE, "workspace needs %zu bytes (16-byte aligned), got %zu", L.bytes,
                        workspace ? workspace_bytes : (size_t)0);
        if (max_batch_blocks > INT32_MAX) return fail(GDN_ERR_INVALID_ARG, "too many blocks in one call");
    }

    // launches, in batches of up to kLaunchSessions sessions
    const int D = d->d_k;
    const int64_t ch = channels(d);
    const int in_bf16 = d->in_dtype == GDN_BF16;
    cudaStream_t cst = (cudaStream_t)stream;
    if (total > 0) {
        const WsLayout L = ws_layout(d, max_batch_blocks);
        // kernel parameters may take up to 32,764 bytes (compute capability 7.0+, CUDA 12.1+)
        static_assert(sizeof(LaunchCommon) <= 32764, "launch parameters must fit the kernel-parameter limit");
        LaunchCommon p;
        fill_common(p, d, xq, xk, xv, g, beta, conv_w, out);
        p.ws_qk = reinterpret_cast<float *>(ws_base(workspace) + L.qk_off);
        p.ws_wu = reinterpret_cast<float *>(ws_base(workspace) + L.wu_off);
        if (in_bf16 && D == 128) {   // input tensor maps of the tcgen05 prologue
            const int64_t rows = cu[n_sessions];
            cudaError_t e = encode_rows_map(&p.tm_q, xq, rows, (int64_t)d->n_qk_heads * D);
            if (e == cudaSuccess) e = encode_rows_map(&p.tm_k, xk, rows, (int64_t)d->n_qk_heads * D);
            if (e == cudaSuccess) e = encode_rows_map(&p.tm_v, xv, rows, (int64_t)d->n_v_heads * D);
            if (e != cudaSuccess) return cuda_fail(e, "input tensor-map encoding");
        }
        for (int i0 = 0; i0 < n_sessions;) {
            int cnt = 0, i = i0, blk = 0;
            for (; i < n_sessions && cnt < gdn::kLaunchSessions; ++i) {
                if (nproc[i] <= 0) continue;
                gdn::SessRef &r = p.s[cnt++];
                r.row0 = cu[i]; r.n = (int32_t)nproc[i]; r.blk0 = blk;
                r.S = sessions[i].S; r.conv = sessions[i].conv;
                r.S0 = prefix ? prefix->S : r.S;
                r.conv0 = prefix ? prefix->conv : r.conv;
                r.S_cap = ckpt ? static_cast<float *>(ckpt[i].S) : nullptr;
                r.conv_cap = ckpt ? ckpt[i].conv : nullptr;
                blk += (int)((nproc[i] + kBlock - 1) / kBlock);
            }
            i0 = i;
            if (cnt == 0) continue;
            p.n_sess = cnt; p.nblk = blk;
            {   // the state kernel starts the longest chains first
                int ord[gdn::kLaunchSessions];
                for (int j = 0; j < cnt; ++j) ord[j] = j;
                std::stable_sort(ord, ord + cnt, [&](int x, int y) { return p.s[x].n > p.s[y].n; });
                for (int j = 0; j < cnt; ++j) p.order[j] = (unsigned char)ord[j];
            }
            cudaError_t e = gdn_device_error_word(&p.err);
            if (e != cudaSuccess) return cuda_fail(e, "device error word lookup");
            int sms = 0;
            if ((e = gdn_sm_count(&sms)) != cudaSuccess) return cuda_fail(e, "SM count");
            // few chains: the one-launch prefill (chains beside the prologue, at least half the SMs for it)
            const int n_fused_chain = cnt * d->n_v_heads * (D / kFusedCols);
            const bool fused = in_bf16 && D == 128 && 2 * n_fused_chain <= sms;
            const int split = in_bf16 && D == 128 && !fused ? tail_split(p, d) : 0;
            if (fused) {
                p.task_block_major = 1;
                auto *flags = reinterpret_cast<unsigned long long *>(ws_base(workspace) + L.flags_off);
                const unsigned long long epoch = ++g_epoch;
                e = launch_k(K_FUSED, cst, [&] { return gdn_launch_prefill_fused(p, ch, flags, epoch, n_fused_chain, cst); });
                p.task_block_major = 0;
            } else if (split > 0) {
                // the call as two parts: blocks [0, split) (prologue, then state pass), then the prologue of
                // the last blocks on the SMs that state pass leaves (running beside it), then their state
                // pass, which continues from the first part's state
                LaunchCommon pa = p, pb = p;
                gdn::SessRef &ra = pa.s[0];
                ra.n = split * kBlock;
                ra.S_cap = nullptr; ra.conv_cap = nullptr;   // the checkpoint is the second part's end
                pa.nblk = split;
                LaunchCommon pt = p;   // the tail prologue: every block of the call in the parameters, tasks of the last
                pt.blk_lo = split;
                gdn::SessRef &rb = pb.s[0];
                rb.row0 += (int64_t)split * kBlock; rb.n -= split * kBlock; rb.blk0 += split;
                rb.S0 = rb.S; rb.conv0 = rb.conv;   // the first part's results
                pb.nblk = p.nblk - split;
                const int cols = gdn_chain_umma_cols(d->n_v_heads, sms);
                const int free_sms = sms - d->n_v_heads * (D / cols);
                e = launch_k(K_PREP, cst, [&] { return gdn_launch_prep_umma(pa, ch, cst); });
                if (e != cudaSuccess) return cuda_fail(e, "prologue/WY kernel");
                e = launch_k(K_STATE, cst, [&] { return gdn_launch_chain_umma(pa, ch, cst, cols); });
                if (e != cudaSuccess) return cuda_fail(e, "state/output kernel");
                e = launch_k(K_PREP_TAIL, cst, [&] { return gdn_launch_prep_umma(pt, ch, cst, free_sms); });
                if (e != cudaSuccess) return cuda_fail(e, "prologue/WY kernel");
                e = launch_k(K_STATE, cst, [&] { return gdn_launch_chain_umma(pb, ch, cst, cols); });
            } else if (in_bf16) {
                // bf16 inputs: tensor-core kernels (d = 128: tcgen05 prologue and state pass over fp16 records;
                // d = 64: the warp-level ones); the state kernel also commits the conv state
                e = launch_k(K_PREP, cst, [&] { return D == 128 ? gdn_launch_prep_umma(p, ch, cst) : gdn_launch_prep_tc(p, D, ch, cst); });
                if (e != cudaSuccess) return cuda_fail(e, "prologue/WY kernel");
                e = launch_k(K_STATE, cst, [&] {
                    return D == 128 ? gdn_launch_chain_umma(p, ch, cst) : gdn_launch_chain_tc(p, D, ch, cst);
                });
            } else {
                // fp32 inputs: fp32 kernels (tighter tolerance)
                e = launch_k(K_PREP, cst, [&] { return gdn_launch_prep(p, D, in_bf16, ch, cst); });
                if (e != cudaSuccess) return cuda_fail(e, "prologue/WY kernel");
                e = launch_k(K_CONV, cst, [&] { return gdn_launch_conv_commit(p, D, in_bf16, ch, cst); });
                if (e != cudaSuccess) return cuda_fail(e, "conv-state commit kernel");
                e = launch_k(K_STATE, cst, [&] { return gdn_launch_state(p, D, cst); });
            }
            if (e != cudaSuccess) return cuda_fail(e, "state/output kernel");
        }
    }
    {   // sessions with nothing to process: a branch becomes a copy of the prefix, a checkpoint a copy of the
        // session's (unchanged) state
        cudaStream_t cst = (cudaStream_t)stream;
        for (int i = 0; i < n_sessions; ++i) {
            if (nproc[i] > 0) continue;
            const gdn_session &from = prefix ? *prefix : sessions[i];
            for (gdn_session *to : {prefix ? &sessions[i] : nullptr, ckpt ? &ckpt[i] : nullptr}) {
                if (!to) continue;
                cudaError_t e = launch_k(K_COPY, cst, [&] {
                    return gdn_launch_copy(to->S, from.S, gdn_state_bytes(d), to->conv, from.conv,
                                           gdn_conv_state_bytes(d), cst);
                });
                if (e != cudaSuccess) return cuda_fail(e, "state copy");
            }
        }
    }
    for (int i = 0; i < n_sessions; ++i) {
        sessions[i].committed = (prefix ? prefix->committed : sessions[i].committed) + nproc[i];
        n_consumed[i] = nproc[i];
        if (ckpt) {
            ckpt[i].committed = sessions[i].committed;
            ckpt[i].tag = tag_of(d);
        }
    }
    return GDN_OK;
}

}  // namespace

GDN_API gdn_status gdn_prefill_varlen(const gdn_layer_desc *d, gdn_session *sessions, int32_t n_sessions,
                                      const int64_t *cu, const void *xq, const void *xk, const void *xv,
                                      const float *g, const float *beta, const void *conv_w, uint32_t flags,
                                      void *out, int64_t *n_consumed, void *workspace, size_t workspace_bytes,
                                      gdn_stream_t stream) {
    return prefill_impl(d, sessions, n_sessions, cu, xq, xk, xv, g, beta, conv_w, flags, out, n_consumed, workspace,
                        workspace_bytes, stream, nullptr, nullptr);
}

GDN_API gdn_status gdn_prefill_varlen_checkpoint(const gdn_layer_desc *d, gdn_session *sessions,
                                                 gdn_session *checkpoints, int32_t n_sessions, const int64_t *cu,
                                                 const void *xq, const void *xk, const void *xv, const float *g,
                                                 const float *beta, const void *conv_w, uint32_t flags, void *out,
                                                 int64_t *n_consumed, void *workspace, size_t workspace_bytes,
                                                 gdn_stream_t stream) {
    if (!checkpoints) return fail(GDN_ERR_INVALID_ARG, "checkpoints is NULL");
    return prefill_impl(d, sessions, n_sessions, cu, xq, xk, xv, g, beta, conv_w, flags, out, n_consumed, workspace,
                        workspace_bytes, stream, nullptr, checkpoints);
}

GDN_API gdn_status gdn_prefill_branches(const gdn_layer_desc *d, const gdn_session *prefix, gdn_session *branches,
                                        int32_t n_branches, const int64_t *cu, const void *xq, const void *xk,
                                        const void *xv, const float *g, const float *beta, const void *conv_w,
                                        uint32_t flags, void *out, int64_t *n_consumed, void *workspace,
                                        size_t workspace_bytes, gdn_stream_t stream) {
    if (!prefix) return fail(GDN_ERR_INVALID_ARG, "prefix is NULL");
    return prefill_impl(d, branches, n_branches, cu, xq, xk, xv, g, beta, conv_w, flags, out, n_consumed, workspace,
                        workspace_bytes, stream, prefix, nullptr);
}

GDN_API gdn_status gdn_prefill_chunks(const gdn_layer_desc *d, gdn_session *session, const void *xq,
                                      const void *xk, const void *xv, const float *g, const float *beta,
                                      const void *conv_w, int64_t n_tokens, uint32_t flags, void *out,
                                      int64_t *n_consumed, void *workspace, size_t workspace_bytes,
                                      gdn_stream_t stream) {
    if (n_tokens < 0) return fail(GDN_ERR_INVALID_ARG, "n_tokens must be >= 0 (got %lld)", (long long)n_tokens);
    const int64_t cu[2] = {0, n_tokens};
    return gdn_prefill_varlen(d, session, 1, cu, xq, xk, xv, g, beta, conv_w, flags, out, n_consumed, workspace,
                              workspace_bytes, stream);
}

GDN_API gdn_status gdn_prefill_chunks_checkpoint(const gdn_layer_desc *d, gdn_session *session, gdn_session *slot,
                                                 const void *xq, const void *xk, const void *xv, const float *g,
                                                 const float *beta, const void *conv_w, int64_t n_tokens,
                                                 uint32_t flags, void *out, int64_t *n_consumed, void *workspace,
                                                 size_t workspace_bytes, gdn_stream_t stream) {
    if (n_tokens < 0) return fail(GDN_ERR_INVALID_ARG, "n_tokens must be >= 0 (got %lld)", (long long)n_tokens);
    const int64_t cu[2] = {0, n_tokens};
    return gdn_prefill_varlen_checkpoint(d, session, slot, 1, cu, xq, xk, xv, g, beta, conv_w, flags, out, n_consumed,
                                         workspace, workspace_bytes, stream);
}

GDN_API gdn_status gdn_state_capture(const gdn_layer_desc *d, const gdn_session *src, gdn_session *slot,
                                     gdn_stream_t stream) {
    gdn_status st = check_desc(d);
    if (st != GDN_OK) return st;
    if ((st = check_state(d, src, "source session", true)) != GDN_OK) return st;
    if (!slot || !slot->S || !slot->conv || !aligned16(slot->S) || !aligned16(slot->conv))
        return fail(GDN_ERR_INVALID_ARG, "slot buffers must be non-NULL and 16-byte aligned");
    if (slot->S == src->S) return fail(GDN_ERR_INVALID_ARG, "slot and source share their buffers");
    slot->committed = -1;  // missing until the copy is enqueued
    slot->tag = 0;
    cudaError_t e = launch_k(K_COPY, (cudaStream_t)stream, [&] {
        return gdn_launch_copy(slot->S, src->S, gdn_state_bytes(d), slot->conv, src->conv,
                               gdn_conv_state_bytes(d), (cudaStream_t)stream);
    });
    if (e != cudaSuccess) return cuda_fail(e, "state capture copy");
    slot->committed = src->committed;
    slot->tag = src->tag;
    return GDN_OK;
}

GDN_API gdn_status gdn_state_restore(const gdn_layer_desc *d, gdn_session *dst, const gdn_session *slot,
                                     gdn_stream_t stream) {
    gdn_status st = check_desc(d);
    if (st != GDN_OK) return st;
    if ((st = check_state(d, slot, "slot", true)) != GDN_OK) return st;
    if ((st = check_state(d, dst, "destination session", false)) != GDN_OK) return st;
    if (slot->S == dst->S) return fail(GDN_ERR_INVALID_ARG, "slot and destination share their buffers");
    cudaError_t e = launch_k(K_COPY, (cudaStream_t)stream, [&] {
        return gdn_launch_copy(dst->S, slot->S, gdn_state_bytes(d), dst->conv, slot->conv,
                               gdn_conv_state_bytes(d), (cudaStream_t)stream);
    });
    if (e != cudaSuccess) return cuda_fail(e, "state restore copy");
    dst->committed = slot->committed;
    return GDN_OK;
}

GDN_API gdn_status gdn_conv_state(const gdn_layer_desc *d, const gdn_session *s, void *out, gdn_stream_t stream) {
    gdn_status st = check_desc(d);
    if (st != GDN_OK) return st;
    if ((st = check_state(d, s, "session", true)) != GDN_OK) return st;
    if (!out) return fail(GDN_ERR_INVALID_ARG, "out is NULL");
    cudaError_t e = cudaMemcpyAsync(out, s->conv, gdn_conv_state_bytes(d), cudaMemcpyDefault, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "conv state copy");
    return GDN_OK;
}

GDN_API gdn_status gdn_decode_step(const gdn_layer_desc *d, gdn_session *sessions, int32_t n, const void *xq,
                                   const void *xk, const void *xv, const float *g, const float *beta,
                                   const void *conv_w, void *out, gdn_stream_t stream) {
    gdn_status st = check_desc(d);
    if (st != GDN_OK) return st;
    if (n < 1 || n > GDN_MAX_SESSIONS)
        return fail(GDN_ERR_INVALID_ARG, "n_sessions must be in [1, %d] (got %d)", GDN_MAX_SESSIONS, n);
    if (!sessions) return fail(GDN_ERR_INVALID_ARG, "sessions is NULL");
    for (int i = 0; i < n; ++i) {
        char what[48];
        snprintf(what, sizeof(what), "session %d", i);
        if ((st = check_state(d, &sessions[i], what, true)) != GDN_OK) return st;
    }
    {
        std::vector<const void *> ptrs(n);
        for (int i = 0; i < n; ++i) ptrs[i] = sessions[i].S;
        std::sort(ptrs.begin(), ptrs.end());
        if (std::adjacent_find(ptrs.begin(), ptrs.end()) != ptrs.end())
            return fail(GDN_ERR_INVALID_ARG, "the sessions of one call must be distinct");
    }
    if (!xq || !xk || !xv || !g || !beta || !conv_w || !out)
        return fail(GDN_ERR_INVALID_ARG, "input / output pointers must be non-NULL");
    if (!aligned16(xq) || !aligned16(xk) || !aligned16(xv) || !aligned16(conv_w) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(g) & 3) || (reinterpret_cast<uintptr_t>(beta) & 3))
        return fail(GDN_ERR_INVALID_ARG, "xq, xk, xv, conv_w, out must be 16-byte aligned; g, beta 4-byte aligned");
    const int D = d->d_k;
    const int64_t ch = channels(d);
    const int in_bf16 = d->in_dtype == GDN_BF16;
    LaunchCommon p;
    fill_common(p, d, xq, xk, xv, g, beta, conv_w, out);
    for (int i0 = 0; i0 < n; i0 += gdn::kLaunchSessions) {
        const int cnt = std::min(n - i0, gdn::kLaunchSessions);
        for (int j = 0; j < cnt; ++j) {
            gdn::SessRef &r = p.s[j];
            r.row0 = i0 + j; r.n = 1; r.blk0 = 0;
            r.S = sessions[i0 + j].S; r.conv = sessions[i0 + j].conv;
            r.S0 = r.S; r.conv0 = r.conv;
        }
        p.n_sess = cnt; p.nblk = 0;
        cudaStream_t cst = (cudaStream_t)stream;
        cudaError_t e = launch_k(K_DECODE, cst, [&] { return gdn_launch_decode(p, D, in_bf16, ch, i0 / gdn::kLaunchSessions, cst); });
        if (e != cudaSuccess) return cuda_fail(e, "decode kernel");
    }
    for (int i = 0; i < n; ++i) sessions[i].committed += 1;
    return GDN_OK;
}

GDN_API gdn_status gdn_gates(const gdn_layer_desc *d, const float *a, const float *b, const float *A_log,
                             const float *dt_bias, int64_t n_tokens, float *g, float *beta, gdn_stream_t stream) {
    gdn_status st = check_desc(d);
    if (st != GDN_OK) return st;
    if (n_tokens < 0 || n_tokens > ((int64_t)1 << 40) / d->n_v_heads)
        return fail(GDN_ERR_INVALID_ARG, "n_tokens out of range (%lld)", (long long)n_tokens);
    if (!a || !b || !A_log || !dt_bias || !g || !beta)
        return fail(GDN_ERR_INVALID_ARG, "a, b, A_log, dt_bias, g, beta must be non-NULL");
    for (const void *q : {(const void *)a, (const void *)b, (const void *)A_log, (const void *)dt_bias,
                          (const void *)g, (const void *)beta})
        if (reinterpret_cast<uintptr_t>(q) & 3) return fail(GDN_ERR_INVALID_ARG, "gate arrays must be 4-byte aligned");
    cudaStream_t cst = (cudaStream_t)stream;
    cudaError_t e = launch_k(K_GATES, cst, [&] {
        return gdn_launch_gates(a, b, A_log, dt_bias, n_tokens * d->n_v_heads, d->n_v_heads, g, beta, cst);
    });
    if (e != cudaSuccess) return cuda_fail(e, "gate kernel");
    return GDN_OK;
}

GDN_API gdn_status gdn_device_status(gdn_stream_t stream) {
    unsigned int word = 0;
    cudaError_t e = gdn_take_device_error(&word, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "device status read");
    if (word & 1u) return fail(GDN_ERR_TIMEOUT, "a kernel gave up waiting for its operand copies");
    return GDN_OK;
}

GDN_API gdn_status gdn_debug_inject_wait_timeout(int32_t enable, int64_t wait_limit) {
    if (!enable) {
        g_skip_first_copy = 0;
        g_wait_limit = kDefaultWaitLimit;
        return GDN_OK;
    }
    if (wait_limit < 1) return fail(GDN_ERR_INVALID_ARG, "wait_limit must be >= 1");
    if (enable != 1 && enable != 2) return fail(GDN_ERR_INVALID_ARG, "enable must be 0, 1 or 2");
    g_skip_first_copy = enable;
    g_wait_limit = wait_limit;
    return GDN_OK;
}

GDN_API const char *gdn_last_error(void) { return g_err; }

GDN_API const char *gdn_status_string(gdn_status s) {
    switch (s) {
        case GDN_OK: return "GDN_OK";
        case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
        case GDN_ERR_SHAPE: return "GDN_ERR_SHAPE";
        case GDN_ERR_OFF_GRID: return "GDN_ERR_OFF_GRID";
        case GDN_ERR_STATE_MISMATCH: return "GDN_ERR_STATE_MISMATCH";
        case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE";
        case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
        case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT";
        case GDN_ERR_NOT_FOUND: return "GDN_ERR_NOT_FOUND";
        case GDN_ERR_IO: return "GDN_ERR_IO";
    }
    return "unknown status";
}
