// gdn_common.cuh -- device helpers shared by the GDN kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gdn.h"

namespace gdn {

// Shapes and scalars every kernel needs, passed by value.
struct Dims {
    int hk, hv, dk, dv, grp;  // grp = hv / hk (v-heads sharing one q/k head)
    int ch;                   // 2*hk*dk + hv*dv
    int chunk;
    int n_slots;
    float q_scale, l2_eps, norm_eps;
    // every bounded wait on the device gives up after wait_ns nanoseconds (gdn_debug_set_wait);
    // `lose` makes chosen launches skip one operand copy so that a wait runs out (tests only)
    unsigned long long wait_ns;
    unsigned lose;
};
constexpr unsigned LOSE_DECODE_STATE_COPY = 1u;   // decode streaming kernel: the first head's state
constexpr unsigned LOSE_CHAIN_OPERAND_COPY = 2u;  // state chain: the first chunk's [-W ; Q'] operand

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// The four conv taps of one channel (row c of the [CH][4] taps, 16-byte aligned base) in one
// vector load, kept raw until every load of a thread has been issued.
template <typename TA> struct TapVec { using type = float4; };
template <> struct TapVec<__nv_bfloat16> { using type = uint2; };
template <typename TA>
__device__ __forceinline__ typename TapVec<TA>::type load_taps(const TA *w, int c) {
    return *reinterpret_cast<const typename TapVec<TA>::type *>(w + (long long)c * 4);
}
__device__ __forceinline__ void taps_f32(const float4 &v, float (&t)[4]) {
    t[0] = v.x; t[1] = v.y; t[2] = v.z; t[3] = v.w;
}
__device__ __forceinline__ void taps_f32(const uint2 &v, float (&t)[4]) {   // bf16 pairs, tap 0 low
    t[0] = __uint_as_float(v.x << 16); t[1] = __uint_as_float(v.x & 0xffff0000u);
    t[2] = __uint_as_float(v.y << 16); t[3] = __uint_as_float(v.y & 0xffff0000u);
}

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }
// SiLU on the approximate-exp and fast-divide intrinsics (relative error about
// 1e-6), for the streaming kernels that apply it to every element.
__device__ __forceinline__ float silu_fast(float x) { return __fdividef(x, 1.0f + __expf(-x)); }
__device__ __forceinline__ float sigmoid_f(float x) { return 1.0f / (1.0f + expf(-x)); }
__device__ __forceinline__ float softplus_f(float x) { return x > 20.0f ? x : log1pf(expf(x)); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Record a device-side fault in the library's error word (never traps).
__device__ __forceinline__ void set_error(unsigned *err, unsigned code) {
    if (err) atomicOr(err, code);
}

// Slot of sequence n: identity without a map; -1 (padding lane) when the map
// says so or the entry is out of range (the latter is also reported).
__device__ __forceinline__ int slot_of(const int32_t *state_idx, int n, int n_slots,
                                       unsigned *err) {
    int s = state_idx ? state_idx[n] : n;
    if (s >= n_slots) {
        set_error(err, GDN_DEVERR_SLOT);
        return -1;
    }
    return s;
}

// Bounds of sequence n, clamped to [0, T] so that malformed cu_seqlens never
// lead to an out-of-range access; malformed input is reported.
__device__ __forceinline__ void seq_bounds(const int32_t *cu, int n, long long T, unsigned *err,
                                           long long &s, long long &e) {
    long long a = cu[n], b = cu[n + 1];
    if (a < 0 || b < a || b > T) {
        set_error(err, GDN_DEVERR_CU_SEQLENS);
        a = a < 0 ? 0 : (a > T ? T : a);
        b = b < a ? a : (b > T ? T : b);
    }
    s = a;
    e = b;
}

}  // namespace gdn

// Launchers implemented by the kernel translation units and called by the ABI.
namespace gdn {
size_t mixer_prefill_ws_bytes(const gdn_config *cfg, long long T, long long n_seqs);
struct ChunkArgs {
    const void *q, *k, *v;
    long long ld_qk, ld_v;
    const float *g, *beta;
    const int32_t *cu_seqlens;
    int n_seqs;
    long long T;
    const float *state_in;
    float *state_out;
    const int32_t *state_idx;
    void *o;
    unsigned flags;
    Dims d;
    unsigned *err;
    // tensor-core path: per-sequence chunk offsets and the [T ; PT] operands
    // (caller workspace, carved by chunk_tc_carve)
    int *chunk_base;
    unsigned char *tp;    // [max_chunks][HV] blocks: [T ; PT] and [-W ; Q'] operands
    unsigned char *kt;    // [max_chunks][HK] blocks: the normalised K (MN-major bf16 hi/lo)
    float *gl;            // G_last of every (chunk, v-head)
    float *kdec;          // [max_chunks][HV][64]: exp(G_last - G_r) of every row
    long long max_chunks;
    // gated RMSNorm fused into the chain's output (then `o` receives y):
    // y = o * rsqrt(mean(o^2) + norm_eps) * w * SiLU(z) per (token, v-head)
    const void *z;        // [T][ld_z] activation dtype
    long long ld_z;
    const float *norm_w;  // [dv]
    float *npart;         // [max_chunks][HV][64 rows][128/32 slices]: per-slice sums of o^2
                          // (null: chunk_tp_kernel leaves no markers there)
};

struct DecodeArgs {
    // fused form: raw x / conv; unfused form: q, k, v post-conv
    const void *x; long long ld_x; const void *conv_w; void *conv_state;
    const void *q, *k, *v; long long ld_qk, ld_v;
    const void *u, *b_logit; long long ld_ub; const float *A_log, *dt_bias;  // fused gates
    const float *g, *beta;                                                   // unfused gates
    const void *z; long long ld_z; const float *norm_w;                      // fused norm
    int n;
    float *state;
    const int32_t *state_idx;
    void *out;  // fused: y; unfused: o
    float *ws;  // fused: per-unit records written by the prep kernel (caller workspace)
    unsigned flags;
    Dims d;
    unsigned *err;
    // multi-token verification (gdn_mixer_verify): k tokens per sequence; the state and conv
    // history after token j go to slot ckpt_idx[n] + j
    int k_tokens;
    const int32_t *ckpt_idx;
    // Q8 state (gdn_mixer_decode_q8): int8 codes [slots][HV][dk][dv], fp32 row scales
    // [slots][HV][dk], and the frame that keys the rounding dither
    int8_t *q8;
    float *q8_scale;
    uint32_t frame;
    __nv_bfloat16 *q8_res;   // error-feedback residual [slots][HV][dk][dv] (null: no feedback)
};
cudaError_t launch_decode_q8(const DecodeArgs &a, bool in_bf16, bool out_bf16, cudaStream_t s);
cudaError_t launch_q8_convert(const Dims &d, const float *state, int8_t *codes, float *scales,
                              __nv_bfloat16 *res, uint32_t frame, bool to_q8, cudaStream_t s);

// Backward of the gated delta rule core (gdn_chunk_states / gdn_chunk_backward).
struct BwdArgs {
    const void *q, *k, *v;
    long long ld_qk, ld_v;
    const float *g, *beta;
    const int32_t *cu_seqlens;
    int n_seqs;
    long long T;
    const float *state_in;        // [slots][HV][dk][dv] or null (zero initial state)
    const int32_t *state_idx;
    float *bnd;                   // [chunks][HV][dk][dv]: the state at every chunk start
    float *pw;                    // [T][HV][2][dv] or null: every token's p = M^T k and w = beta (v - a p)
    const float *d_o;             // [T][HV*dv]
    const float *d_state_out;     // [slots][HV][dk][dv] or null
    float *dq, *dk;               // [T][ld_dqk], q/k head kh at column kh*dk
    long long ld_dqk;
    float *dv;                    // [T][HV*dv]
    float *dg, *dbeta;            // [T][HV]
    float *d_state_in;            // [slots][HV][dk][dv] or null
    Dims d;
    unsigned *err;
    // workspace (bwd_carve)
    int *chunk_base;              // [n_seqs + 1]
    float *scratch;               // [n_seqs][HV][slices][segments][chunk/2][dk][32]: states before the even tokens
    float *gsplit;                // [n_seqs][HV][segments-1][dk][dv]: dL/dS entering each later segment
    float *pq, *pk;               // [T][HV][slices][dk]: the parts of dq, dk from each 32-column slice
    float *pda, *pda2, *pdb;      // [T][HV][slices]: the parts of <GM, M>, dw . p and dw . r
};
size_t bwd_ws_bytes(const Dims &d, long long T, long long n_seqs, bool states_only);
void bwd_carve(BwdArgs &a, void *ws, bool states_only);
cudaError_t launch_backward(const BwdArgs &a, bool in_bf16, bool states_only, cudaStream_t s);

// Per-(sequence, q/k head) record the fused decode's prep kernel writes and its
// streaming kernel reads (floats): normalised q and k, conv'd v and SiLU(z) of
// the unit's G v-heads, the gates a and beta, k.q, and the state slot.
struct DecRec {
    int q, k, v, z, ga, gb, kq, slot, size;
    __host__ __device__ DecRec(int dk, int dv, int g) {
        q = 0; k = dk; v = 2 * dk; z = v + g * dv; ga = z + g * dv; gb = ga + g; kq = gb + g;
        slot = kq + 1;
        size = (slot + 1 + 3) & ~3;      // 16-byte multiple
    }
};
size_t decode_ws_bytes(const Dims &d, long long n_seqs);
// gdn_mixer_verify: a record per (sequence, q/k head, token); ws_bytes for n_seqs * k tokens
constexpr int kMaxVerify = 8;
cudaError_t launch_verify(const DecodeArgs &a, bool in_bf16, bool out_bf16, cudaStream_t s);

cudaError_t launch_gate_prep(const Dims &d, bool act_bf16, const void *u, const void *b,
                             long long ld_ub, long long T, const float *A_log,
                             const float *dt_bias, float *g, float *beta, cudaStream_t s);
// Gates computed by the conv kernel (the mixer prefill): u, b_logit [T][ld_ub] in the activation
// dtype; g, beta [T][HV] fp32.  g == nullptr: none.
struct GateArgs {
    const void *u, *b;
    long long ld_ub;
    const float *A_log, *dt_bias;
    float *g, *beta;
};
cudaError_t launch_conv_prefill(const Dims &d, bool act_bf16, const void *x, long long ld_x,
                                const int32_t *cu, int n_seqs, long long T, const void *w,
                                const void *conv_state, const int32_t *state_idx, void *out,
                                bool out_bf16, unsigned *err, cudaStream_t s,
                                const GateArgs *gates = nullptr);
// Snapshot / restore / reset of state slots (gdn_state_copy); the history
// words per slot assume CH * 3 * element size is a multiple of 16 bytes.
cudaError_t launch_state_copy(const Dims &d, bool act_bf16, const float *src_state,
                              const void *src_conv, int n_src, float *dst_state, void *dst_conv,
                              int n_dst, const int32_t *src_idx, const int32_t *dst_idx, int n,
                              unsigned *err, cudaStream_t s);
cudaError_t launch_conv_state_update(const Dims &d, bool act_bf16, const void *x,
                                     long long ld_x, const int32_t *cu, int n_seqs, long long T,
                                     void *conv_state, const int32_t *state_idx, unsigned *err,
                                     cudaStream_t s);
cudaError_t launch_conv_step(const Dims &d, bool act_bf16, const void *x, long long ld_x, int n,
                             const void *w, void *conv_state, const int32_t *state_idx,
                             void *out, bool out_bf16, unsigned *err, cudaStream_t s);
cudaError_t launch_gated_rmsnorm(const Dims &d, bool act_bf16, const void *o, bool o_bf16,
                                 const void *z, long long ld_z, const float *w, long long T,
                                 void *y, bool y_bf16, cudaStream_t s);
cudaError_t launch_chunk_simt(const ChunkArgs &a, bool in_bf16, bool o_bf16, cudaStream_t s);
bool chunk_tc_supported(const Dims &d);
long long chunk_tc_max_chunks(long long T, long long n_seqs);
size_t chunk_tc_ws_bytes(const Dims &d, long long T, long long n_seqs);
void chunk_tc_carve(ChunkArgs &a, void *ws);
cudaError_t launch_chunk_tc(const ChunkArgs &a, bool in_bf16, bool o_bf16, int dvs, bool fuse_norm,
                            cudaStream_t s);
// Streaming multiprocessors of the current device (cached per device).
int sm_count();
cudaError_t launch_decode(const DecodeArgs &a, bool fused, bool in_bf16, bool out_bf16,
                          cudaStream_t s);
}  // namespace gdn
