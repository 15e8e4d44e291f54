// gdn_elementwise.cu -- gate prep, causal conv1d (prefill and one-token step)
// with SiLU, conv-history update, and the gated RMSNorm.
//
// All of these are HBM-bound streaming kernels: channel-contiguous threads so
// that every warp reads and writes whole 64- or 128-byte rows, fp32 math,
// grids sized to the problem (they are short and launch-count matters more
// than occupancy tuning here).
#include "gdn_common.cuh"

namespace gdn {

// ------------------------------------------------------------------ gates
// g = -exp(A_log[h]) * softplus(u + dt_bias[h]);  beta = sigmoid(b_logit).
template <typename TIn>
__global__ void gate_prep_kernel(Dims d, const TIn *u, const TIn *b, long long ld_ub, long long T,
                                 const float *A_log, const float *dt_bias, float *g,
                                 float *beta) {
    long long total = T * d.hv;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        long long t = e / d.hv;
        int h = (int)(e - t * d.hv);
        float uu = to_f32(u[t * ld_ub + h]) + dt_bias[h];
        g[e] = -expf(A_log[h]) * softplus_f(uu);
        beta[e] = sigmoid_f(to_f32(b[t * ld_ub + h]));
    }
}

cudaError_t launch_gate_prep(const Dims &d, bool act_bf16, const void *u, const void *b,
                             long long ld_ub, long long T, const float *A_log,
                             const float *dt_bias, float *g, float *beta, cudaStream_t s) {
    long long total = T * d.hv;
    if (total == 0) return cudaSuccess;
    int blocks = (int)((total + 255) / 256);
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (act_bf16)
        gate_prep_kernel<<<blocks, 256, 0, s>>>(d, (const __nv_bfloat16 *)u,
                                                (const __nv_bfloat16 *)b, ld_ub, T, A_log,
                                                dt_bias, g, beta);
    else
        gate_prep_kernel<<<blocks, 256, 0, s>>>(d, (const float *)u, (const float *)b, ld_ub, T,
                                                A_log, dt_bias, g, beta);
    return cudaGetLastError();
}

// ------------------------------------------------------------ conv prefill
// Each thread owns 8 consecutive channels (one 16-byte row segment of bf16
// input) for CONV_TT consecutive tokens, sliding a 3-token window in
// registers: one vector load and one or two vector stores per token.  Taps
// before a sequence start come from its history slot (zero without one).
// Outputs only: the history is replaced afterwards by
// conv_state_update_kernel, so no CTA can overwrite a history another CTA
// still has to read.
constexpr int CONV_TT = 64;
constexpr int CONV_B = 4;      // tokens whose loads are issued together
constexpr int CONV_NT = 128;
constexpr int CONV_V = 8;

__device__ __forceinline__ void load8f(const float *p, float *v) {
    const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8f(const __nv_bfloat16 *p, float *v) {
    const uint4 u = *reinterpret_cast<const uint4 *>(p);
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
    }
}
__device__ __forceinline__ void store8f(float *p, const float *v) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void store8f(__nv_bfloat16 *p, const float *v) {
    __nv_bfloat162 h[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    *reinterpret_cast<uint4 *>(p) = *reinterpret_cast<const uint4 *>(h);
}

template <typename TA, typename TO>
__global__ void __launch_bounds__(CONV_NT, 4)
    conv_prefill_kernel(Dims d, const TA *x, long long ld_x, const int32_t *cu, int n_seqs,
                        long long T, const TA *w, const TA *conv_state,
                        const int32_t *state_idx, TO *out, unsigned *err, GateArgs ga) {
    const int c0 = (blockIdx.y * CONV_NT + threadIdx.x) * CONV_V;
    const long long t0 = (long long)blockIdx.x * CONV_TT;
    if (ga.g && blockIdx.y == 0 && t0 < T) {
        // the gates of this CTA's tokens (the mixer prefill folds gate_prep_kernel in here):
        // the same expressions, element for element
        const long long tend = t0 + CONV_TT < T ? t0 + CONV_TT : T;
        for (long long e = t0 * d.hv + threadIdx.x; e < tend * d.hv; e += CONV_NT) {
            const long long t = e / d.hv;
            const int h = (int)(e - t * d.hv);
            const float uu = to_f32(((const TA *)ga.u)[t * ga.ld_ub + h]) + ga.dt_bias[h];
            ga.g[e] = -expf(ga.A_log[h]) * softplus_f(uu);
            ga.beta[e] = sigmoid_f(to_f32(((const TA *)ga.b)[t * ga.ld_ub + h]));
        }
    }
    if (c0 >= d.ch || t0 >= T) return;
    float wv[CONV_V][4];
    {
        float wf[4 * CONV_V];
#pragma unroll
        for (int i = 0; i < 4; ++i) load8f(w + (long long)c0 * 4 + 8 * i, wf + 8 * i);
#pragma unroll
        for (int i = 0; i < CONV_V; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j) wv[i][j] = wf[4 * i + j];
    }
    // sequence containing t0: last n with cu[n] <= t0 (empty sequences skipped below)
    int lo = 0, hi = n_seqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= t0) lo = mid; else hi = mid - 1;
    }
    int n = lo;
    long long s, e;
    seq_bounds(cu, n, T, err, s, e);
    while (t0 >= e && n + 1 < n_seqs) { ++n; seq_bounds(cu, n, T, err, s, e); }
    int slot = slot_of(state_idx, n, d.n_slots, err);
    // the three taps before token t of the current sequence (window[0] oldest)
    float win[3][CONV_V];
    auto fill_window = [&](long long t) {
        float hist[3 * CONV_V];
        const bool has_hist = conv_state && slot >= 0;
        if (has_hist) {
            const TA *hp = conv_state + ((long long)slot * d.ch + c0) * 3;
#pragma unroll
            for (int i = 0; i < 3; ++i) load8f(hp + 8 * i, hist + 8 * i);
        }
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const long long tt = t - 3 + j;
            if (tt >= s) {
                load8f(x + tt * ld_x + c0, win[j]);
            } else {
                const int hj = (int)(tt - s + 3);     // in [0, 3) since t >= s
#pragma unroll
                for (int i = 0; i < CONV_V; ++i) {
                    float hv = 0.f;
#pragma unroll
                    for (int q = 0; q < 3; ++q)
                        if (q == hj) hv = hist[3 * i + q];
                    win[j][i] = has_hist ? hv : 0.f;
                }
            }
        }
    };
    fill_window(t0);
    const long long t_end = t0 + CONV_TT < T ? t0 + CONV_TT : T;
    // one output token of the current sequence, sliding the window
    auto step = [&](const float (&cur)[CONV_V], long long t) {
        float o[CONV_V];
#pragma unroll
        for (int i = 0; i < CONV_V; ++i) {
            const float acc = wv[i][0] * win[0][i] + wv[i][1] * win[1][i] + wv[i][2] * win[2][i] +
                              wv[i][3] * cur[i];
            o[i] = silu_fast(acc);
            win[0][i] = win[1][i];
            win[1][i] = win[2][i];
            win[2][i] = cur[i];
        }
        store8f(out + t * d.ch + c0, o);
    };
    for (long long tb = t0; tb < t_end; tb += CONV_B) {
        if (tb + CONV_B <= t_end && tb + CONV_B <= e) {
            // CONV_B tokens inside the current sequence: all their loads in flight at once
            float cur[CONV_B][CONV_V];
#pragma unroll
            for (int b = 0; b < CONV_B; ++b) load8f(x + (tb + b) * ld_x + c0, cur[b]);
#pragma unroll
            for (int b = 0; b < CONV_B; ++b) step(cur[b], tb + b);
        } else {
            const long long tend = tb + CONV_B < t_end ? tb + CONV_B : t_end;
            for (long long t = tb; t < tend; ++t) {
                if (t >= e && n + 1 < n_seqs) {   // the next sequence starts here
                    while (t >= e && n + 1 < n_seqs) {
                        ++n;
                        seq_bounds(cu, n, T, err, s, e);
                    }
                    slot = slot_of(state_idx, n, d.n_slots, err);
                    fill_window(t);
                }
                float cur[CONV_V];
                load8f(x + t * ld_x + c0, cur);
                step(cur, t);
            }
        }
    }
}

// New history of each active sequence = its last three raw inputs, reaching
// into the old history when the sequence is shorter than three tokens.
template <typename TA>
__global__ void conv_state_update_kernel(Dims d, const TA *x, long long ld_x, const int32_t *cu,
                                         int n_seqs, long long T, TA *conv_state,
                                         const int32_t *state_idx, unsigned *err) {
    int n = blockIdx.y;
    int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= d.ch || n >= n_seqs) return;
    long long s, e;
    seq_bounds(cu, n, T, err, s, e);
    if (n == n_seqs - 1 && c == 0 && cu[n_seqs] != T) set_error(err, GDN_DEVERR_CU_SEQLENS);
    int slot = slot_of(state_idx, n, d.n_slots, err);
    if (slot < 0) return;
    TA *h = conv_state + ((long long)slot * d.ch + c) * 3;
    long long L = e - s;
    TA old[3] = {h[0], h[1], h[2]};
    TA nw[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        long long tt = e - 3 + j;
        nw[j] = (tt >= s) ? x[tt * ld_x + c] : old[L + j];
    }
    h[0] = nw[0];
    h[1] = nw[1];
    h[2] = nw[2];
}

cudaError_t launch_conv_prefill(const Dims &d, bool act_bf16, const void *x, long long ld_x,
                                const int32_t *cu, int n_seqs, long long T, const void *w,
                                const void *conv_state, const int32_t *state_idx, void *out,
                                bool out_bf16, unsigned *err, cudaStream_t s, const GateArgs *gates) {
    const GateArgs ga = gates ? *gates : GateArgs{};
    if (T == 0 || n_seqs == 0) return cudaSuccess;
    dim3 grid((unsigned)((T + CONV_TT - 1) / CONV_TT), (d.ch + CONV_NT * CONV_V - 1) / (CONV_NT * CONV_V));
#define GDN_CONV(TA, TO)                                                                   \
    conv_prefill_kernel<TA, TO><<<grid, CONV_NT, 0, s>>>(                                   \
        d, (const TA *)x, ld_x, cu, n_seqs, T, (const TA *)w, (const TA *)conv_state,       \
        state_idx, (TO *)out, err, ga)
    if (act_bf16) {
        if (out_bf16) GDN_CONV(__nv_bfloat16, __nv_bfloat16); else GDN_CONV(__nv_bfloat16, float);
    } else {
        if (out_bf16) GDN_CONV(float, __nv_bfloat16); else GDN_CONV(float, float);
    }
#undef GDN_CONV
    return cudaGetLastError();
}

cudaError_t launch_conv_state_update(const Dims &d, bool act_bf16, const void *x,
                                     long long ld_x, const int32_t *cu, int n_seqs, long long T,
                                     void *conv_state, const int32_t *state_idx, unsigned *err,
                                     cudaStream_t s) {
    if (!conv_state || n_seqs == 0) return cudaSuccess;
    dim3 grid((d.ch + 255) / 256, n_seqs);
    if (act_bf16)
        conv_state_update_kernel<<<grid, 256, 0, s>>>(d, (const __nv_bfloat16 *)x, ld_x, cu,
                                                      n_seqs, T, (__nv_bfloat16 *)conv_state,
                                                      state_idx, err);
    else
        conv_state_update_kernel<<<grid, 256, 0, s>>>(d, (const float *)x, ld_x, cu, n_seqs, T,
                                                      (float *)conv_state, state_idx, err);
    return cudaGetLastError();
}

// ------------------------------------------------------------- conv step
// One token per sequence; each (sequence, channel) history is owned by one
// thread, so the in-place shift needs no ordering.
template <typename TA, typename TO>
__global__ void conv_step_kernel(Dims d, const TA *x, long long ld_x, int n_seqs, const TA *w,
                                 TA *conv_state, const int32_t *state_idx, TO *out,
                                 unsigned *err) {
    int n = blockIdx.y;
    int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= d.ch || n >= n_seqs) return;
    int slot = slot_of(state_idx, n, d.n_slots, err);
    float xv = to_f32(x[(long long)n * ld_x + c]);
    float h0 = 0.f, h1 = 0.f, h2 = 0.f;
    TA *h = nullptr;
    if (slot >= 0) {
        h = conv_state + ((long long)slot * d.ch + c) * 3;
        h0 = to_f32(h[0]); h1 = to_f32(h[1]); h2 = to_f32(h[2]);
    }
    float acc = to_f32(w[c * 4 + 0]) * h0 + to_f32(w[c * 4 + 1]) * h1 +
                to_f32(w[c * 4 + 2]) * h2 + to_f32(w[c * 4 + 3]) * xv;
    out[(long long)n * d.ch + c] = from_f32<TO>(silu_f(acc));
    if (h) {
        TA t1 = h[1], t2 = h[2];
        h[0] = t1;
        h[1] = t2;
        h[2] = x[(long long)n * ld_x + c];
    }
}

cudaError_t launch_conv_step(const Dims &d, bool act_bf16, const void *x, long long ld_x, int n,
                             const void *w, void *conv_state, const int32_t *state_idx,
                             void *out, bool out_bf16, unsigned *err, cudaStream_t s) {
    if (n == 0) return cudaSuccess;
    dim3 grid((d.ch + 255) / 256, n);
#define GDN_STEP(TA, TO)                                                                    \
    conv_step_kernel<TA, TO><<<grid, 256, 0, s>>>(d, (const TA *)x, ld_x, n, (const TA *)w, \
                                                  (TA *)conv_state, state_idx, (TO *)out, err)
    if (act_bf16) {
        if (out_bf16) GDN_STEP(__nv_bfloat16, __nv_bfloat16); else GDN_STEP(__nv_bfloat16, float);
    } else {
        if (out_bf16) GDN_STEP(float, __nv_bfloat16); else GDN_STEP(float, float);
    }
#undef GDN_STEP
    return cudaGetLastError();
}

// ------------------------------------------------------------ gated norm
// One warp per (token, v-head) row of dv values, lane l holding the dv/32
// consecutive values l*dv/32 ..: y = o*rsqrt(mean(o^2)+eps)*w*SiLU(z).
template <int PER, typename T>
__device__ __forceinline__ void loadv(const T *p, float *v) {
#pragma unroll
    for (int i = 0; i < PER; ++i) v[i] = to_f32(p[i]);
}
template <>
__device__ __forceinline__ void loadv<4, float>(const float *p, float *v) {
    const float4 a = *reinterpret_cast<const float4 *>(p);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
}
template <>
__device__ __forceinline__ void loadv<4, __nv_bfloat16>(const __nv_bfloat16 *p, float *v) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
    const float2 a = __bfloat1622float2(h[0]), b = __bfloat1622float2(h[1]);
    v[0] = a.x; v[1] = a.y; v[2] = b.x; v[3] = b.y;
}
template <int PER, typename T>
__device__ __forceinline__ void storev(T *p, const float *v) {
#pragma unroll
    for (int i = 0; i < PER; ++i) p[i] = from_f32<T>(v[i]);
}
template <>
__device__ __forceinline__ void storev<4, float>(float *p, const float *v) {
    *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
template <>
__device__ __forceinline__ void storev<4, __nv_bfloat16>(__nv_bfloat16 *p, const float *v) {
    __nv_bfloat162 h[2] = {__floats2bfloat162_rn(v[0], v[1]), __floats2bfloat162_rn(v[2], v[3])};
    *reinterpret_cast<uint2 *>(p) = *reinterpret_cast<const uint2 *>(h);
}

template <int DV, typename TO_IN, typename TZ, typename TY>
__global__ void gated_rmsnorm_kernel(Dims d, const TO_IN *o, const TZ *z, long long ld_z,
                                     const float *w, long long T, TY *y) {
    constexpr int PER = DV / 32;
    const long long rows = T * d.hv;
    const int lane = threadIdx.x & 31;
    const long long warp = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    float wv[PER];
    loadv<PER>(w + lane * PER, wv);
    for (long long r = warp; r < rows; r += nwarps) {
        const long long t = r / d.hv;
        const int h = (int)(r - t * d.hv);
        float ov[PER], zv[PER];
        loadv<PER>(o + r * DV + lane * PER, ov);
        loadv<PER>(z + t * ld_z + (long long)h * DV + lane * PER, zv);
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < PER; ++i) ss += ov[i] * ov[i];
        ss = warp_sum(ss);
        const float rs = rsqrtf(ss / (float)DV + d.norm_eps);
        float yv[PER];
#pragma unroll
        for (int i = 0; i < PER; ++i) yv[i] = ov[i] * rs * wv[i] * silu_fast(zv[i]);
        storev<PER>(y + r * DV + lane * PER, yv);
    }
}

template <int DV>
static void launch_norm_dv(const Dims &d, bool act_bf16, const void *o, bool o_bf16,
                           const void *z, long long ld_z, const float *w, long long T, void *y,
                           bool y_bf16, cudaStream_t s) {
    long long rows = T * d.hv;
    int blocks = (int)((rows + 7) / 8);
    if (blocks > 152 * 32) blocks = 152 * 32;
#define GDN_NORM(TOI, TZ, TY)                                                              \
    gated_rmsnorm_kernel<DV, TOI, TZ, TY><<<blocks, 256, 0, s>>>(d, (const TOI *)o,        \
                                                                 (const TZ *)z, ld_z, w, T, \
                                                                 (TY *)y)
    if (act_bf16) {
        if (o_bf16) {
            if (y_bf16) GDN_NORM(__nv_bfloat16, __nv_bfloat16, __nv_bfloat16);
            else GDN_NORM(__nv_bfloat16, __nv_bfloat16, float);
        } else {
            if (y_bf16) GDN_NORM(float, __nv_bfloat16, __nv_bfloat16);
            else GDN_NORM(float, __nv_bfloat16, float);
        }
    } else {
        if (o_bf16) {
            if (y_bf16) GDN_NORM(__nv_bfloat16, float, __nv_bfloat16);
            else GDN_NORM(__nv_bfloat16, float, float);
        } else {
            if (y_bf16) GDN_NORM(float, float, __nv_bfloat16);
            else GDN_NORM(float, float, float);
        }
    }
#undef GDN_NORM
}

cudaError_t launch_gated_rmsnorm(const Dims &d, bool act_bf16, const void *o, bool o_bf16,
                                 const void *z, long long ld_z, const float *w, long long T,
                                 void *y, bool y_bf16, cudaStream_t s) {
    if (T == 0) return cudaSuccess;
    switch (d.dv) {
        case 32: launch_norm_dv<32>(d, act_bf16, o, o_bf16, z, ld_z, w, T, y, y_bf16, s); break;
        case 64: launch_norm_dv<64>(d, act_bf16, o, o_bf16, z, ld_z, w, T, y, y_bf16, s); break;
        case 128: launch_norm_dv<128>(d, act_bf16, o, o_bf16, z, ld_z, w, T, y, y_bf16, s); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace gdn
