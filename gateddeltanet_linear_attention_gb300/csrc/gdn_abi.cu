// gdn_abi.cu -- the extern "C" entry points of include/gdn.h: host-side
// argument validation (before any launch), workspace carving, dispatch to the
// kernels, and the device error word.
#include <cmath>
#include <atomic>
#include <mutex>

#include "gdn_common.cuh"

namespace {

// Device-side fault word: kernels OR GDN_DEVERR_* bits into it, never trap.
__device__ unsigned g_gdn_error_word;

constexpr int kMaxDevices = 64;
unsigned *g_err_ptr[kMaxDevices];
std::mutex g_err_mu;

// Address of the error word on the current device (resolved once per device).
gdn_status error_word(unsigned **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GDN_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_err_mu);
    if (!g_err_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_gdn_error_word) != cudaSuccess) return GDN_ERR_CUDA;
        g_err_ptr[dev] = (unsigned *)p;
    }
    *out = g_err_ptr[dev];
    return GDN_OK;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Limit of every bounded wait on the device, and the test hook that makes a
// launch lose one operand copy (gdn_debug_set_wait); read at each call.
std::atomic<unsigned long long> g_wait_ns{2000000000ull};
std::atomic<unsigned> g_lose{0u};

// Largest sequence count a call accepts (one grid dimension per sequence).
constexpr int kMaxSeqs = 65535;

bool valid_dtype(gdn_dtype t) { return t == GDN_BF16 || t == GDN_FP32; }

// Validate the configuration and derive the kernel-side dimensions.
gdn_status check_cfg(const gdn_config *c, gdn::Dims *d) {
    if (!c) return GDN_ERR_INVALID_ARG;
    if (c->hk <= 0 || c->hv <= 0 || c->dk <= 0 || c->dv <= 0 || c->chunk <= 0 ||
        c->n_slots < 0 || !valid_dtype(c->act))
        return GDN_ERR_INVALID_ARG;
    if (!(std::isfinite(c->q_scale) && std::isfinite(c->l2_eps) && std::isfinite(c->norm_eps)) ||
        c->l2_eps < 0.f || c->norm_eps < 0.f)
        return GDN_ERR_INVALID_ARG;
    if (c->hv % c->hk != 0) return GDN_ERR_INVALID_ARG;
    const int grp = c->hv / c->hk;
    if (grp != 1 && grp != 2 && grp != 4) return GDN_ERR_UNSUPPORTED;
    if (c->dk != c->dv || (c->dk != 32 && c->dk != 64 && c->dk != 128)) return GDN_ERR_UNSUPPORTED;
    if (c->chunk != 16 && c->chunk != 64) return GDN_ERR_UNSUPPORTED;
    long long ch = 2LL * c->hk * c->dk + (long long)c->hv * c->dv;
    if (ch > (1LL << 22)) return GDN_ERR_UNSUPPORTED;
    d->hk = c->hk; d->hv = c->hv; d->dk = c->dk; d->dv = c->dv; d->grp = grp;
    d->ch = (int)ch; d->chunk = c->chunk; d->n_slots = c->n_slots;
    d->q_scale = c->q_scale; d->l2_eps = c->l2_eps; d->norm_eps = c->norm_eps;
    d->wait_ns = g_wait_ns.load();
    d->lose = g_lose.load();
    return GDN_OK;
}

// A row-strided [rows][ld] view with `width` used elements per row, rows
// 16-byte aligned (vector / bulk loads).
bool valid_view(const void *p, long long ld, long long width) {
    return p && aligned16(p) && ld >= width && ld % 8 == 0;
}

// A narrow row-strided view read element by element (u, b_logit: HV columns).
bool valid_narrow_view(const void *p, long long ld, long long width) {
    return p && ((uintptr_t)p & 3u) == 0 && ld >= width;
}

gdn_status launch_status(cudaError_t e) { return e == cudaSuccess ? GDN_OK : GDN_ERR_CUDA; }

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

struct PrefillWs {
    float *xa, *g, *beta, *o;
    void *chunk;   // tensor-core chunk workspace (chunk map + [T ; PT] operands), or NULL
};

// The chunked rule: bf16-activation configurations with dk = dv = 128 and
// 64-token chunks run on the tensor cores (split-bf16 operands); everything
// else, and the fp32-activation mode, runs the exact fp32 SIMT kernel.
bool uses_tc(const gdn::Dims &d, bool act_bf16) { return act_bf16 && gdn::chunk_tc_supported(d); }

size_t chunk_ws_bytes(const gdn::Dims &d, bool act_bf16, long long T, long long n_seqs) {
    return uses_tc(d, act_bf16) ? gdn::chunk_tc_ws_bytes(d, T, n_seqs) : 0;
}

// The tensor-core path launches one CTA per (chunk, q/k head) in a 1-D grid (checked with
// HV >= HK, which also bounds the per-(chunk, v-head) workspace indices).
bool tc_grid_fits(const gdn::Dims &d, bool act_bf16, long long T, long long n_seqs) {
    return !uses_tc(d, act_bf16) || gdn::chunk_tc_max_chunks(T, n_seqs) * d.hv <= 0x7fffffffLL;
}

// The fp32 o between the chunked rule and the gated norm exists only on the
// SIMT path; the tensor-core chain applies the norm itself.
size_t prefill_o_bytes(const gdn::Dims &d, bool act_bf16, long long T) {
    return uses_tc(d, act_bf16) ? 0 : align256((size_t)(T > 0 ? T : 0) * d.hv * d.dv * 4);
}

size_t prefill_ws_bytes(const gdn::Dims &d, bool act_bf16, long long T, long long n_seqs) {
    size_t t = (size_t)(T > 0 ? T : 0);
    return align256(t * d.ch * 4) + 2 * align256(t * d.hv * 4) + prefill_o_bytes(d, act_bf16, T) +
           align256(chunk_ws_bytes(d, act_bf16, T, n_seqs));
}

PrefillWs carve_prefill(const gdn::Dims &d, bool act_bf16, long long T, long long n_seqs, void *ws) {
    size_t t = (size_t)T;
    char *p = (char *)ws;
    PrefillWs w;
    w.xa = (float *)p; p += align256(t * d.ch * 4);
    w.g = (float *)p; p += align256(t * d.hv * 4);
    w.beta = (float *)p; p += align256(t * d.hv * 4);
    w.o = (float *)p; p += prefill_o_bytes(d, act_bf16, T);
    w.chunk = chunk_ws_bytes(d, act_bf16, T, n_seqs) ? (void *)p : nullptr;
    return w;
}

// Each tensor-core CTA owns a 32-column slice of one head's state; the chunk
// workspace `ws` must already be carved into `a` (chunk_tc_carve).
cudaError_t launch_chunk(const gdn::ChunkArgs &a, bool act_bf16, bool in_bf16, bool o_bf16,
                         cudaStream_t s, bool fuse_norm = false) {
    if (uses_tc(a.d, act_bf16)) return gdn::launch_chunk_tc(a, in_bf16, o_bf16, 32, fuse_norm, s);
    return gdn::launch_chunk_simt(a, in_bf16, o_bf16, s);
}

}  // namespace

namespace gdn {
// Bytes of the fused prefill's intermediates alone (0 for an invalid configuration).
size_t mixer_prefill_ws_bytes(const gdn_config *cfg, long long T, long long n_seqs) {
    Dims d;
    if (check_cfg(cfg, &d) != GDN_OK || T < 0 || n_seqs < 0) return 0;
    return prefill_ws_bytes(d, cfg->act == GDN_BF16, T, n_seqs);
}

int sm_count() {
    static int cached[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
    if (!cached[dev]) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
            v = 148;
        cached[dev] = v;
    }
    return cached[dev];
}
}  // namespace gdn

extern "C" {

const char *gdn_status_string(gdn_status s) {
    switch (s) {
        case GDN_OK: return "ok";
        case GDN_ERR_INVALID_ARG: return "invalid argument";
        case GDN_ERR_UNSUPPORTED: return "unsupported configuration";
        case GDN_ERR_WORKSPACE: return "workspace missing or too small";
        case GDN_ERR_CUDA: return "CUDA error";
        case GDN_ERR_DEVICE: return "device-side fault reported";
    }
    return "unknown status";
}

size_t gdn_workspace_size(const gdn_config *cfg, int64_t max_tokens, int32_t max_seqs) {
    gdn::Dims d;
    if (check_cfg(cfg, &d) != GDN_OK || max_tokens < 0 || max_seqs < 0) return 0;
    const size_t pre = prefill_ws_bytes(d, cfg->act == GDN_BF16, max_tokens, max_seqs),
                 dec = gdn::decode_ws_bytes(d, max_seqs);
    return (pre > dec ? pre : dec) + 256;
}

gdn_status gdn_gate_prep(const gdn_config *cfg, const void *u, const void *b_logit, int64_t ld_ub,
                         int64_t T, const float *A_log, const float *dt_bias, float *g,
                         float *beta, void *stream) {
    gdn::Dims d;
    gdn_status st = check_cfg(cfg, &d);
    if (st != GDN_OK) return st;
    if (T < 0) return GDN_ERR_INVALID_ARG;
    if (T == 0) return GDN_OK;
    if (!valid_narrow_view(u, ld_ub, d.hv) || !valid_narrow_view(b_logit, ld_ub, d.hv) || !A_log || !dt_bias ||
        !g || !beta)
        return GDN_ERR_INVALID_ARG;
    return launch_status(gdn::launch_gate_prep(d, cfg->act == GDN_BF16, u, b_logit, ld_ub, T,
                                               A_log, dt_bias, g, beta, (cudaStream_t)stream));
}

gdn_status gdn_conv1d_prefill(const gdn_config *cfg, const void *x, int64_t ld_x,
                              const int32_t *cu_seqlens, int32_t n_seqs, int64_t T,
                              const void *w, void *conv_state, const int32_t *state_idx,
                              void *out, gdn_dtype out_dtype, void *stream) {
    gdn::Dims d;
    gdn_status st = check_cfg(cfg, &d);
    if (st != GDN_OK) return st;
    if (T < 0 || n_seqs < 0 || !valid_dtype(out_dtype)) return GDN_ERR_INVALID_ARG;
    if (n_seqs > kMaxSeqs) return GDN_ERR_UNSUPPORTED;
    if (n_seqs == 0 || T == 0) {
        if (T != 0) return GDN_ERR_INVALID_ARG;
        if (n_seqs == 0) return GDN_OK;
    }
    if (!cu_seqlens || !w || !aligned16(w) || !out || !aligned16(out) ||
        (T > 0 && !valid_view(x, ld_x, d.ch)))
        return GDN_ERR_INVALID_ARG;
    if (conv_state && !aligned16(conv_state)) return GDN_ERR_INVALID_ARG;
    if (conv_state && d.n_slots == 0) return GDN_ERR_INVALID_ARG;
    unsigned *err = nullptr;
    if ((st = error_word(&err)) != GDN_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    const bool bf = cfg->act == GDN_BF16;
    cudaError_t e = gdn::launch_conv_prefill(d, bf, x, ld_x, cu_seqlens, n_seqs, T, w, conv_state,
                                             state_idx, out, out_dtype == GDN_BF16, err, s);
    if (e == cudaSuccess)
        e = gdn::launch_conv_state_update(d, bf, x, ld_x, cu_seqlens, n_seqs, T, conv_state,
                                          state_idx, err, s);
    return launch_status(e);
}

gdn_status gdn_conv1d_step(const gdn_config *cfg, const void *x, int64_t ld_x, int32_t n,
                           const void *w, void *conv_state, const int32_t *state_idx, void *out,
                           gdn_dtype out_dtype, void *stream) {
    gdn::Dims d;
    gdn_status st = check_cfg(cfg, &d);
    if (st != GDN_OK) return st;
    if (n < 0 || !valid_dtype(out_dtype)) return GDN_ERR_INVALID_ARG;
    if (n > kMaxSeqs) return GDN_ERR_UNSUPPORTED;
    if (n == 0) return GDN_OK;
    if (!valid_view(x, ld_x, d.ch) || !w || !conv_state || !aligned16(conv_state) || !out ||
        d.n_slots == 0)
        return GDN_ERR_INVALID_ARG;
    unsigned *err = nullptr;
    if ((st = error_word(&err)) != GDN_OK) return st;
    return launch_status(gdn::launch_conv_step(d, cfg->act == GDN_BF16, x, ld_x, n, w, conv_state,
                                               state_idx, out, out_dtype == GDN_BF16, err,
                                               (cudaStream_t)stream));
}

gdn_status gdn_chunk_prefill(const gdn_config *cfg, const void *q, const void *k, int64_t ld_qk,
                             const void *v, int64_t ld_v, gdn_dtype in_dtype, const float *g,
                             const float *beta, const int32_t *cu_seqlens, int32_t n_seqs,
                             int64_t T, const float *state_in, float *state_out,
                             const int32_t *state_idx, void *o, gdn_dtype o_dtype, uint32_t flags,
                             void *workspace, size_t workspace_bytes, void *stream) {
    gdn::Dims d;
    gdn_status st = check_cfg(cfg, &d);
    if (st != GDN_OK) return st;
    if (T < 0 || n_seqs < 0 || !valid_dtype(in_dtype) || !valid_dtype(o_dtype) ||
        (flags & ~GDN_FLAG_L2NORM_QK))
        return GDN_ERR_INVALID_ARG;
    if (n_seqs > kMaxSeqs) return GDN_ERR_UNSUPPORTED;
    if (n_seqs == 0) return T == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
    if (!cu_seqlens || !g || !beta || !o || !aligned16(o)) return GDN_ERR_INVALID_ARG;
    if (T > 0 && (!valid_view(q, ld_qk, (long long)d.hk * d.dk) ||
                  !valid_view(k, ld_qk, (long long)d.hk * d.dk) ||
                  !valid_view(v, ld_v, (long long)d.hv * d.dv)))
        return GDN_ERR_INVALID_ARG;
    if ((state_in && !aligned16(state_in)) || (state_out && !aligned16(state_out)))
        return GDN_ERR_INVALID_ARG;
    if ((state_in || state_out) && d.n_slots == 0) return GDN_ERR_INVALID_ARG;
    const bool bf = cfg->act == GDN_BF16;
    if (!tc_grid_fits(d, bf, T, n_seqs)) return GDN_ERR_UNSUPPORTED;
    const size_t need = chunk_ws_bytes(d, bf, T, n_seqs);
    if (need && (!workspace || !aligned16(workspace) || workspace_bytes < need))
        return GDN_ERR_WORKSPACE;
    unsigned *err = nullptr;
    if ((st = error_word(&err)) != GDN_OK) return st;
    gdn::ChunkArgs a = {};
    a.q = q; a.k = k; a.v = v; a.ld_qk = ld_qk; a.ld_v = ld_v; a.g = g; a.beta = beta;
    a.cu_seqlens = cu_seqlens; a.n_seqs = n_seqs; a.T = T; a.state_in = state_in;
    a.state_out = state_out; a.state_idx = state_idx; a.o = o; a.flags = flags; a.d = d;
    a.err = err;
    if (need) gdn::chunk_tc_carve(a, workspace);
    return launch_status(launch_chunk(a, bf, in_dtype == GDN_BF16,
                                      o_dtype == GDN_BF16, (cudaStream_t)stream));
}

gdn_status gdn_recurrent_decode(const gdn_config *cfg, const void *q, const void *k, int64_t ld_qk,
                                const void *v, int64_t ld_v, gdn_dtype in_dtype, const float *g,
                                const float *beta, int32_t n, float *state,
                                const int32_t *state_idx, void *o, gdn_dtype o_dtype,
                                uint32_t flags, void *stream) {
    gdn::Dims d;
    gdn_status st = check_cfg(cfg, &d);
    if (st != GDN_OK) return st;
    if (n < 0 || !valid_dtype(in_dtype) || !valid_dtype(o_dtype) || (flags & ~GDN_FLAG_L2NORM_QK))
        return GDN_ERR_INVALID_ARG;
    if (n > kMaxSeqs) return GDN_ERR_UNSUPPORTED;
    if (n == 0) return GDN_OK;
    if (!valid_view(q, ld_qk, (long long)d.hk * d.dk) ||
        !valid_view(k, ld_qk, (long long)d.hk * d.dk) ||
        !valid_view(v, ld_v, (long long)d.hv * d.dv) || !g || !beta || !state ||
        !aligned16(state) || !o || d.n_slots == 0)
        return GDN_ERR_INVALID_ARG;
    unsigned *err = nullptr;
    if ((st = error_word(&err)) != GDN_OK) return st;
    gdn::DecodeArgs a = {};
    a.q = q; a.k = k; a.v = v; a.ld_qk = ld_qk; a.ld_v = ld_v; a.g = g; a.beta = beta;
    a.n = n; a.state = state; a.state_idx = state_idx; a.out = o; a.flags = flags; a.d = d;
    a.err = err;
    return launch_status(gdn::launch_decode(a, false, in_dtype == GDN_BF16, o_dtype == GDN_BF16,
                                            (cudaStream_t)stream));
}

gdn_status gdn_gated_rmsnorm(const gdn_config *cfg, const void *o, gdn_dtype o_dtype,
                             const void *z, int64_t ld_z, const float *w, int64_t T, void *y,
                             gdn_dtype y_dtype, void *stream) {
    gdn::Dims d;
    gdn_status st = check_cfg(cfg, &d);
    if (st != GDN_OK) return st;
    if (T < 0 || !valid_dtype(o_dtype) || !valid_dtype(y_dtype)) return GDN_ERR_INVALID_ARG;
    if (T == 0) return GDN_OK;
    if (!o || !aligned16(o) || !valid_view(z, ld_z, (long long)d.hv * d.dv) || !w ||
        !aligned16(w) || !y || !aligned16(y))
        return GDN_ERR_INVALID_ARG;
    return launch_status(gdn::launch_gated_rmsnorm(d, cfg->act == GDN_BF16, o, o_dtype == GDN_BF16,
                                                   z, ld_z, w, T, y, y_dtype == GDN_BF16,
                                                   (cudaStream_t)stream));
}

// Validation shared by the fused entry points.
// decode: one token per sequence, the state updated in place (q8: the fp32 state pointers must
// be NULL, the state lives in the caller's Q8 pool)
static gdn_status check_mixer_io(const gdn::Dims &d, const gdn_mixer_io *io, bool decode,
                                 bool q8 = false) {
    if (!io || io->n_seqs < 0 || io->T < 0 || !valid_dtype(io->y_dtype)) return GDN_ERR_INVALID_ARG;
    if (io->n_seqs > kMaxSeqs) return GDN_ERR_UNSUPPORTED;
    if (decode && io->T != io->n_seqs) return GDN_ERR_INVALID_ARG;
    if (io->T == 0) return GDN_OK;
    if (!valid_view(io->x, io->ld_x, d.ch) || !valid_view(io->z, io->ld_z, (long long)d.hv * d.dv) ||
        !valid_narrow_view(io->u, io->ld_ub, d.hv) || !valid_narrow_view(io->b_logit, io->ld_ub, d.hv) ||
        !io->conv_w || !aligned16(io->conv_w) || !io->A_log || !io->dt_bias || !io->norm_w ||
        !aligned16(io->norm_w) || !io->y || !aligned16(io->y))
        return GDN_ERR_INVALID_ARG;
    if (!decode && !io->cu_seqlens) return GDN_ERR_INVALID_ARG;
    if ((io->state_in && !aligned16(io->state_in)) || (io->state_out && !aligned16(io->state_out)) ||
        (io->conv_state && !aligned16(io->conv_state)))
        return GDN_ERR_INVALID_ARG;
    if ((io->state_in || io->state_out || io->conv_state) && d.n_slots == 0)
        return GDN_ERR_INVALID_ARG;
    if (decode && !q8 && (!io->state_in || io->state_out != io->state_in || !io->conv_state))
        return GDN_ERR_INVALID_ARG;
    if (q8 && (io->state_in || io->state_out || !io->conv_state || d.n_slots == 0))
        return GDN_ERR_INVALID_ARG;
    return GDN_OK;
}

gdn_status gdn_mixer_prefill(const gdn_config *cfg, const gdn_mixer_io *io, void *workspace,
                             size_t workspace_bytes, void *stream) {
    gdn::Dims d;
    gdn_status st = check_cfg(cfg, &d);
    if (st != GDN_OK) return st;
    if ((st = check_mixer_io(d, io, false)) != GDN_OK) return st;
    if (io->n_seqs == 0) return io->T == 0 ? GDN_OK : GDN_ERR_INVALID_ARG;
    unsigned *err = nullptr;
    cudaStream_t s = (cudaStream_t)stream;
    if (io->T == 0) {
        // only empty sequences: the state passes through (written when out != in)
        if (!io->state_out || io->state_out == io->state_in) return GDN_OK;
        if ((st = error_word(&err)) != GDN_OK) return st;
        gdn::ChunkArgs a = {};
        a.cu_seqlens = io->cu_seqlens; a.n_seqs = io->n_seqs; a.T = 0;
        a.state_in = io->state_in; a.state_out = io->state_out; a.state_idx = io->state_idx;
        a.o = io->y; a.flags = GDN_FLAG_L2NORM_QK; a.d = d; a.err = err;
        return launch_status(launch_chunk(a, cfg->act == GDN_BF16, false, false, s));
    }
    const bool bf = cfg->act == GDN_BF16;
    if (!tc_grid_fits(d, bf, io->T, io->n_seqs)) return GDN_ERR_UNSUPPORTED;
    if (!workspace || !aligned16(workspace) ||
        workspace_bytes < prefill_ws_bytes(d, bf, io->T, io->n_seqs))
        return GDN_ERR_WORKSPACE;
    if ((st = error_word(&err)) != GDN_OK) return st;
    PrefillWs w = carve_prefill(d, bf, io->T, io->n_seqs, workspace);
    // the gates come out of the conv kernel (one launch fewer)
    const gdn::GateArgs ga = {io->u, io->b_logit, io->ld_ub, io->A_log, io->dt_bias, w.g, w.beta};
    cudaError_t e = gdn::launch_conv_prefill(d, bf, io->x, io->ld_x, io->cu_seqlens, io->n_seqs,
                                             io->T, io->conv_w, io->conv_state, io->state_idx,
                                             w.xa, false, err, s, &ga);
    if (e == cudaSuccess)
        e = gdn::launch_conv_state_update(d, bf, io->x, io->ld_x, io->cu_seqlens, io->n_seqs,
                                          io->T, io->conv_state, io->state_idx, err, s);
    if (e == cudaSuccess) {
        gdn::ChunkArgs a = {};
        a.q = w.xa;
        a.k = w.xa + (long long)d.hk * d.dk;
        a.v = w.xa + 2LL * d.hk * d.dk;
        a.ld_qk = d.ch; a.ld_v = d.ch; a.g = w.g; a.beta = w.beta;
        a.cu_seqlens = io->cu_seqlens; a.n_seqs = io->n_seqs; a.T = io->T;
        a.state_in = io->state_in; a.state_out = io->state_out; a.state_idx = io->state_idx;
        a.flags = GDN_FLAG_L2NORM_QK; a.d = d; a.err = err;
        if (uses_tc(d, bf)) {
            // the chain applies the gated norm to its output rows and writes y
            gdn::chunk_tc_carve(a, w.chunk);
            a.o = io->y; a.z = io->z; a.ld_z = io->ld_z; a.norm_w = io->norm_w;
            e = launch_chunk(a, bf, false, io->y_dtype == GDN_BF16, s, true);
        } else {
            a.o = w.o;
            e = launch_chunk(a, bf, false, false, s);
            if (e == cudaSuccess)
                e = gdn::launch_gated_rmsnorm(d, bf, w.o, false, io->z, io->ld_z, io->norm_w, io->T,
                                              io->y, io->y_dtype == GDN_BF16, s);
        }
    }
    return launch_status(e);
}

gdn_status gdn_mixer_decode(const gdn_config *cfg, const gdn_mixer_io *io, void *workspace,
                            size_t workspace_bytes, void *stream) {
    gdn::Dims d;
    gdn_status st = check_cfg(cfg, &d);
    if (st != GDN_OK) return st;
    if ((st = check_mixer_io(d, io, true)) != GDN_OK) return st;
    if (io->n_seqs == 0) return GDN_OK;
    if (!workspace || !aligned16(workspace) ||
        workspace_bytes < gdn::decode_ws_bytes(d, io->n_seqs))
        return GDN_ERR_WORKSPACE;
    unsigned *err = nullptr;
    if ((st = error_word(&err)) != GDN_OK) return st;
    gdn::DecodeArgs a = {};
    a.x = io->x; a.ld_x = io->ld_x; a.conv_w = io->conv_w; a.conv_state = io->conv_state;
    a.u = io->u; a.b_logit = io->b_logit; a.ld_ub = io->ld_ub; a.A_log = io->A_log;
    a.dt_bias = io->dt_bias; a.z = io->z; a.ld_z = io->ld_z; a.norm_w = io->norm_w;
    a.n = io->n_seqs; a.state = io->state_out; a.state_idx = io->state_idx; a.out = io->y;
    a.ws = (float *)workspace;
    a.flags = GDN_FLAG_L2NORM_QK; a.d = d; a.err = err;
    return launch_status(gdn::launch_decode(a, true, cfg->act == GDN_BF16,
                                            io->y_dtype == GDN_BF16, (cudaStream_t)stream));
}

gdn_status gdn_state_copy(const gdn_config *cfg, const float *src_state, const void *src_conv,
                          int32_t n_src_slots, float *dst_state, void *dst_conv,
                          int32_t n_dst_slots, const int32_t *src_idx, const int32_t *dst_idx,
                          int32_t n, void *stream) {
    gdn::Dims d;
    gdn_status st = check_cfg(cfg, &d);
    if (st != GDN_OK) return st;
    if (n < 0 || n > kMaxSeqs || n_src_slots < 0 || n_dst_slots < 0) return GDN_ERR_INVALID_ARG;
    if (n == 0 || (!dst_state && !dst_conv)) return GDN_OK;
    if (!src_idx || !dst_idx) return GDN_ERR_INVALID_ARG;
    if ((src_state && !aligned16(src_state)) || (dst_state && !aligned16(dst_state)) ||
        (src_conv && !aligned16(src_conv)) || (dst_conv && !aligned16(dst_conv)))
        return GDN_ERR_INVALID_ARG;
    if ((long long)d.ch * 3 * (cfg->act == GDN_BF16 ? 2 : 4) % 16 != 0) return GDN_ERR_UNSUPPORTED;
    unsigned *err = nullptr;
    if ((st = error_word(&err)) != GDN_OK) return st;
    return launch_status(gdn::launch_state_copy(d, cfg->act == GDN_BF16, src_state, src_conv,
                                                n_src_slots, dst_state, dst_conv, n_dst_slots,
                                                src_idx, dst_idx, n, err, (cudaStream_t)stream));
}

gdn_status gdn_mixer_verify(const gdn_config *cfg, const gdn_mixer_io *io, int32_t k,
                            const int32_t *ckpt_idx, void *workspace, size_t workspace_bytes,
                            void *stream) {
    gdn::Dims d;
    gdn_status st = check_cfg(cfg, &d);
    if (st != GDN_OK) return st;
    if (!io || k < 1 || k > gdn::kMaxVerify || io->n_seqs < 0) return GDN_ERR_INVALID_ARG;
    if (io->T != (int64_t)io->n_seqs * k) return GDN_ERR_INVALID_ARG;
    // the token-level checks of the one-token decode, applied to the n*k rows
    gdn_mixer_io one = *io;
    one.T = one.n_seqs = (int32_t)((int64_t)io->n_seqs * k > kMaxSeqs ? kMaxSeqs + 1 : io->n_seqs * k);
    if ((st = check_mixer_io(d, &one, true)) != GDN_OK) return st;
    if (io->n_seqs == 0) return GDN_OK;
    if (!ckpt_idx) return GDN_ERR_INVALID_ARG;
    (void)workspace;          // unused: the records live in shared memory
    (void)workspace_bytes;
    unsigned *err = nullptr;
    if ((st = error_word(&err)) != GDN_OK) return st;
    gdn::DecodeArgs a = {};
    a.x = io->x; a.ld_x = io->ld_x; a.conv_w = io->conv_w; a.conv_state = io->conv_state;
    a.u = io->u; a.b_logit = io->b_logit; a.ld_ub = io->ld_ub; a.A_log = io->A_log;
    a.dt_bias = io->dt_bias; a.z = io->z; a.ld_z = io->ld_z; a.norm_w = io->norm_w;
    a.n = io->n_seqs; a.state = io->state_out; a.state_idx = io->state_idx; a.out = io->y;
    a.flags = GDN_FLAG_L2NORM_QK; a.d = d; a.err = err;
    a.k_tokens = k; a.ckpt_idx = ckpt_idx;
    return launch_status(gdn::launch_verify(a, cfg->act == GDN_BF16, io->y_dtype == GDN_BF16,
                                            (cudaStream_t)stream));
}

size_t gdn_backward_workspace_size(const gdn_config *cfg, int64_t max_tokens, int32_t max_seqs) {
    gdn::Dims d;
    if (check_cfg(cfg, &d) != GDN_OK || max_tokens < 0 || max_seqs < 0) return 0;
    return gdn::bwd_ws_bytes(d, max_tokens, max_seqs, false) + 256;
}

// Arguments both backward entry points share: k, v, gates and the batch.
static gdn_status check_bwd_common(const gdn::Dims &d, const void *k, int64_t ld_qk, const void *v,
                                   int64_t ld_v, gdn_dtype in_dtype, const float *g,
                                   const float *beta, const int32_t *cu_seqlens, int32_t n_seqs,
                                   int64_t T) {
    if (n_seqs < 0 || T < 0 || !valid_dtype(in_dtype)) return GDN_ERR_INVALID_ARG;
    if (n_seqs > kMaxSeqs) return GDN_ERR_UNSUPPORTED;
    if (T == 0) return GDN_OK;
    if (n_seqs == 0 || !cu_seqlens) return GDN_ERR_INVALID_ARG;
    if (!valid_view(k, ld_qk, (long long)d.hk * d.dk) || !valid_view(v, ld_v, (long long)d.hv * d.dv) ||
        !g || !aligned16(g) || !beta || !aligned16(beta))
        return GDN_ERR_INVALID_ARG;
    return GDN_OK;
}

gdn_status gdn_chunk_states(const gdn_config *cfg, const void *k, int64_t ld_qk, const void *v,
                            int64_t ld_v, gdn_dtype in_dtype, const float *g, const float *beta,
                            const int32_t *cu_seqlens, int32_t n_seqs, int64_t T,
                            const float *state_in, const int32_t *state_idx, float *boundary_states,
                            float *token_pw, void *workspace, size_t workspace_bytes, void *stream) {
    gdn::Dims d;
    gdn_status st = check_cfg(cfg, &d);
    if (st != GDN_OK) return st;
    if ((st = check_bwd_common(d, k, ld_qk, v, ld_v, in_dtype, g, beta, cu_seqlens, n_seqs, T)) != GDN_OK)
        return st;
    if (T == 0) return GDN_OK;
    if (!boundary_states || !aligned16(boundary_states) || (state_in && !aligned16(state_in)) ||
        (token_pw && !aligned16(token_pw)))
        return GDN_ERR_INVALID_ARG;
    if (state_in && d.n_slots == 0) return GDN_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) || workspace_bytes < gdn::bwd_ws_bytes(d, T, n_seqs, true))
        return GDN_ERR_WORKSPACE;
    unsigned *err = nullptr;
    if ((st = error_word(&err)) != GDN_OK) return st;
    gdn::BwdArgs a = {};
    a.k = k; a.v = v; a.ld_qk = ld_qk; a.ld_v = ld_v; a.g = g; a.beta = beta;
    a.cu_seqlens = cu_seqlens; a.n_seqs = n_seqs; a.T = T; a.state_in = state_in;
    a.state_idx = state_idx; a.bnd = boundary_states; a.pw = token_pw; a.d = d; a.err = err;
    gdn::bwd_carve(a, workspace, true);
    return launch_status(gdn::launch_backward(a, in_dtype == GDN_BF16, true, (cudaStream_t)stream));
}

gdn_status gdn_chunk_backward(const gdn_config *cfg, const void *q, const void *k, int64_t ld_qk,
                              const void *v, int64_t ld_v, gdn_dtype in_dtype, const float *g,
                              const float *beta, const int32_t *cu_seqlens, int32_t n_seqs, int64_t T,
                              const int32_t *state_idx, const float *boundary_states,
                              const float *token_pw, const float *d_o, const float *d_state_out,
                              float *dq, float *dk,
                              int64_t ld_dqk, float *dv, float *dg, float *dbeta, float *d_state_in,
                              void *workspace, size_t workspace_bytes, void *stream) {
    gdn::Dims d;
    gdn_status st = check_cfg(cfg, &d);
    if (st != GDN_OK) return st;
    if ((st = check_bwd_common(d, k, ld_qk, v, ld_v, in_dtype, g, beta, cu_seqlens, n_seqs, T)) != GDN_OK)
        return st;
    if ((d_state_out && !aligned16(d_state_out)) || (d_state_in && !aligned16(d_state_in)) ||
        (token_pw && !aligned16(token_pw)))
        return GDN_ERR_INVALID_ARG;
    if ((d_state_out || d_state_in) && d.n_slots == 0) return GDN_ERR_INVALID_ARG;
    if (T == 0) return GDN_OK;
    if (!valid_view(q, ld_qk, (long long)d.hk * d.dk) || !boundary_states || !aligned16(boundary_states) ||
        !d_o || !aligned16(d_o) || !dq || !dk || !aligned16(dq) || !aligned16(dk) ||
        ld_dqk < (long long)d.hk * d.dk || !dv || !aligned16(dv) || !dg || !aligned16(dg) || !dbeta ||
        !aligned16(dbeta))
        return GDN_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) || workspace_bytes < gdn::bwd_ws_bytes(d, T, n_seqs, false))
        return GDN_ERR_WORKSPACE;
    unsigned *err = nullptr;
    if ((st = error_word(&err)) != GDN_OK) return st;
    gdn::BwdArgs a = {};
    a.q = q; a.k = k; a.v = v; a.ld_qk = ld_qk; a.ld_v = ld_v; a.g = g; a.beta = beta;
    a.cu_seqlens = cu_seqlens; a.n_seqs = n_seqs; a.T = T; a.state_idx = state_idx;
    a.bnd = const_cast<float *>(boundary_states); a.pw = const_cast<float *>(token_pw);
    a.d_o = d_o; a.d_state_out = d_state_out;
    a.dq = dq; a.dk = dk; a.ld_dqk = ld_dqk; a.dv = dv; a.dg = dg; a.dbeta = dbeta;
    a.d_state_in = d_state_in; a.d = d; a.err = err;
    gdn::bwd_carve(a, workspace, false);
    return launch_status(gdn::launch_backward(a, in_dtype == GDN_BF16, false, (cudaStream_t)stream));
}

gdn_status gdn_state_to_q8(const gdn_config *cfg, const float *state, int8_t *codes, float *scales,
                           void *residual, uint32_t frame, void *stream) {
    gdn::Dims d;
    gdn_status st = check_cfg(cfg, &d);
    if (st != GDN_OK) return st;
    if (!state || !codes || !scales || !aligned16(state) || !aligned16(codes) || !aligned16(scales) ||
        (residual && !aligned16(residual)))
        return GDN_ERR_INVALID_ARG;
    if (d.n_slots == 0) return GDN_OK;
    return launch_status(gdn::launch_q8_convert(d, state, codes, scales, (__nv_bfloat16 *)residual, frame,
                                                true, (cudaStream_t)stream));
}

gdn_status gdn_state_from_q8(const gdn_config *cfg, const int8_t *codes, const float *scales,
                             float *state, void *stream) {
    gdn::Dims d;
    gdn_status st = check_cfg(cfg, &d);
    if (st != GDN_OK) return st;
    if (!state || !codes || !scales || !aligned16(state) || !aligned16(codes) || !aligned16(scales))
        return GDN_ERR_INVALID_ARG;
    if (d.n_slots == 0) return GDN_OK;
    return launch_status(gdn::launch_q8_convert(d, state, const_cast<int8_t *>(codes),
                                                const_cast<float *>(scales), nullptr, 0u, false,
                                                (cudaStream_t)stream));
}

gdn_status gdn_mixer_decode_q8(const gdn_config *cfg, const gdn_mixer_io *io, int8_t *codes,
                               float *scales, void *residual, uint32_t frame, void *workspace,
                               size_t workspace_bytes, void *stream) {
    gdn::Dims d;
    gdn_status st = check_cfg(cfg, &d);
    if (st != GDN_OK) return st;
    if ((st = check_mixer_io(d, io, true, true)) != GDN_OK) return st;
    if (io->n_seqs == 0) return GDN_OK;
    if (!codes || !scales || !aligned16(codes) || !aligned16(scales) || (residual && !aligned16(residual)))
        return GDN_ERR_INVALID_ARG;
    if (!workspace || !aligned16(workspace) ||
        workspace_bytes < gdn::decode_ws_bytes(d, io->n_seqs))
        return GDN_ERR_WORKSPACE;
    unsigned *err = nullptr;
    if ((st = error_word(&err)) != GDN_OK) return st;
    gdn::DecodeArgs a = {};
    a.x = io->x; a.ld_x = io->ld_x; a.conv_w = io->conv_w; a.conv_state = io->conv_state;
    a.u = io->u; a.b_logit = io->b_logit; a.ld_ub = io->ld_ub; a.A_log = io->A_log;
    a.dt_bias = io->dt_bias; a.z = io->z; a.ld_z = io->ld_z; a.norm_w = io->norm_w;
    a.n = io->n_seqs; a.state_idx = io->state_idx; a.out = io->y;
    a.ws = (float *)workspace;
    a.flags = GDN_FLAG_L2NORM_QK; a.d = d; a.err = err;
    a.q8 = codes; a.q8_scale = scales; a.frame = frame; a.q8_res = (__nv_bfloat16 *)residual;
    return launch_status(gdn::launch_decode_q8(a, cfg->act == GDN_BF16, io->y_dtype == GDN_BF16,
                                               (cudaStream_t)stream));
}

gdn_status gdn_debug_set_wait(uint64_t wait_ns, uint32_t lose) {
    if (wait_ns == 0 || wait_ns > 60000000000ull || (lose & ~3u)) return GDN_ERR_INVALID_ARG;
    g_wait_ns.store(wait_ns);
    g_lose.store(lose);
    return GDN_OK;
}

gdn_status gdn_device_error(void *stream, uint32_t *code) {
    if (!code) return GDN_ERR_INVALID_ARG;
    *code = 0;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return GDN_ERR_CUDA;
    unsigned v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_gdn_error_word, sizeof(v)) != cudaSuccess) return GDN_ERR_CUDA;
    if (v && cudaMemcpyToSymbol(g_gdn_error_word, &zero, sizeof(zero)) != cudaSuccess)
        return GDN_ERR_CUDA;
    *code = v;
    return v ? GDN_ERR_DEVICE : GDN_OK;
}

}  // extern "C"
