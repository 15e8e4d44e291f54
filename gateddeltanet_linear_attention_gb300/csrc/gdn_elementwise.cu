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
// One thread per channel, CONV_TT consecutive tokens per CTA row.  Token t of
// sequence n (start s) reads taps x[t-3..t]; taps before s come from the
// sequence's history slot (zero without one).  Outputs only: the history is
// replaced afterwards by conv_state_update_kernel, so no CTA can overwrite a
// history another CTA still has to read.
constexpr int CONV_TT = 32;
constexpr int CONV_NT = 128;

template <typename TA, typename TO>
__global__ void __launch_bounds__(CONV_NT)
    conv_prefill_kernel(Dims d, const TA *x, long long ld_x, const int32_t *cu, int n_seqs,
                        long long T, const TA *w, const TA *conv_state,
                        const int32_t *state_idx, TO *out, unsigned *err) {
    int c = blockIdx.y * CONV_NT + threadIdx.x;
    long long t0 = (long long)blockIdx.x * CONV_TT;
    if (c >= d.ch || t0 >= T) return;
    float w0 = to_f32(w[c * 4 + 0]), w1 = to_f32(w[c * 4 + 1]), w2 = to_f32(w[c * 4 + 2]),
          w3 = to_f32(w[c * 4 + 3]);
    // sequence containing t0: last n with cu[n] <= t0 (first of equal starts skipped below)
    int lo = 0, hi = n_seqs - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= t0) lo = mid; else hi = mid - 1;
    }
    int n = lo;
    long long s, e;
    seq_bounds(cu, n, T, err, s, e);
    while (t0 >= e && n + 1 < n_seqs) { ++n; seq_bounds(cu, n, T, err, s, e); }
    int slot = slot_of(state_idx, n, d.n_slots, err);
    long long t_end = t0 + CONV_TT < T ? t0 + CONV_TT : T;
    for (long long t = t0; t < t_end; ++t) {
        while (t >= e && n + 1 < n_seqs) {
            ++n;
            seq_bounds(cu, n, T, err, s, e);
            slot = slot_of(state_idx, n, d.n_slots, err);
        }
        float tap[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            long long tt = t - 3 + j;
            float val = 0.0f;
            if (tt >= s) {
                val = to_f32(x[tt * ld_x + c]);
            } else if (conv_state && slot >= 0 && tt >= s - 3) {
                val = to_f32(conv_state[((long long)slot * d.ch + c) * 3 + (tt - s + 3)]);
            }
            tap[j] = val;
        }
        float acc = w0 * tap[0] + w1 * tap[1] + w2 * tap[2] + w3 * tap[3];
        out[t * d.ch + c] = from_f32<TO>(silu_f(acc));
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
                                bool out_bf16, unsigned *err, cudaStream_t s) {
    if (T == 0 || n_seqs == 0) return cudaSuccess;
    dim3 grid((unsigned)((T + CONV_TT - 1) / CONV_TT), (d.ch + CONV_NT - 1) / CONV_NT);
#define GDN_CONV(TA, TO)                                                                   \
    conv_prefill_kernel<TA, TO><<<grid, CONV_NT, 0, s>>>(                                   \
        d, (const TA *)x, ld_x, cu, n_seqs, T, (const TA *)w, (const TA *)conv_state,       \
        state_idx, (TO *)out, err)
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
// One warp per (token, v-head) row of dv values: y = o*rsqrt(mean(o^2)+eps)*w*SiLU(z).
template <int DV, typename TO_IN, typename TZ, typename TY>
__global__ void gated_rmsnorm_kernel(Dims d, const TO_IN *o, const TZ *z, long long ld_z,
                                     const float *w, long long T, TY *y) {
    constexpr int PER = DV / 32;
    long long rows = T * d.hv;
    int lane = threadIdx.x & 31;
    long long warp = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
    long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    for (long long r = warp; r < rows; r += nwarps) {
        long long t = r / d.hv;
        int h = (int)(r - t * d.hv);
        const TO_IN *orow = o + r * DV;
        const TZ *zrow = z + t * ld_z + (long long)h * DV;
        float ov[PER], ss = 0.f;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            ov[i] = to_f32(orow[lane + 32 * i]);
            ss += ov[i] * ov[i];
        }
        ss = warp_sum(ss);
        float rs = rsqrtf(ss / (float)DV + d.norm_eps);
        TY *yrow = y + r * DV;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            int j = lane + 32 * i;
            yrow[j] = from_f32<TY>(ov[i] * rs * w[j] * silu_f(to_f32(zrow[j])));
        }
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
