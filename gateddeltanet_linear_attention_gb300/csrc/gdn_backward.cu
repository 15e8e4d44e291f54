// gdn_backward.cu -- backward of the gated delta rule core from retained
// chunk-boundary states (hyperflare core-design, the training plan: a
// training step retains activations and GDN chunk-boundary states, and the
// backward has one entry per region, the GDN core among them).
//
// With the state held as M = S^T (dk x dv), per token of one v-head
// (a = exp(g)):
//   forward   p = M^T k,  w = beta (v - a p),  M' = a M + k w^T,  o = M'^T q
//   backward, GM = dL/dM' (carried from the later tokens):
//     GM += q do^T;            dq = M' do
//     dw = GM^T k;             dk = GM w + M dp
//     dv = beta dw;            dbeta = dw . (v - a p)
//     dp = -a beta dw;         da = <GM, M> - beta dw . p;   dg = a da
//     GM <- a GM + k dp^T      (= dL/dM of the state before the token)
// Every quantity the recurrences carry (M, GM, p, w, dw, dp) is per state
// column, so each CTA owns one 32-column slice of a head's state; only the
// outputs that sum over columns (dq and dk: row sums; da: <GM, M> and dw . p;
// dbeta: dw . r) come out as per-slice parts that a last kernel adds up.
// The kernels:
//  - bwd_states_kernel (gdn_chunk_states): one CTA per (sequence, v-head,
//    slice), the forward over the sequence with the slice of M in registers
//    (thread: one float4 column group over RPT rows, 8 lanes per 128-byte row
//    segment), writing it at every chunk start, and optionally every token's p
//    and w: what a training forward retains.  It takes the tokens in pairs: one
//    pass over M gives M^T k of both, and the pair's k . k fixes the second
//    token's p;
//  - bwd_gm_kernel (gdn_chunk_backward, first): dL/dS at the segment
//    boundaries of the walk below, carried back without the forward states,
//    also in token pairs;
//  - bwd_kernel: one CTA per (sequence, v-head, slice, segment), the chunks in
//    reverse: the forward of the chunk from its boundary state (from the
//    retained p and w when given: no sums), keeping the state before every even
//    token in the workspace, then the tokens in reverse with GM in registers.
//    Column sums go through one shared-memory pass, row sums through shuffles
//    among the lanes that hold the row;
//  - bwd_group_sum_kernel adds the slices and the v-heads of each q/k head
//    (dq, dk) and the slices of each v-head (dg = a (<GM, M> - beta dw . p),
//    dbeta).
#include <type_traits>

#include "gdn_common.cuh"

namespace gdn {

namespace {

// DV here is the slice width (32 columns, one warp for the per-column steps); a thread holds
// 4 columns of RPT consecutive rows (rows rg*RPT .. rg*RPT + RPT-1 for row group rg), so that
// its RPT values of a staged k or q row come in one vector load.
constexpr int BWD_DVS = 32;
template <int DK, int DV>
struct BwdCfg {
    static constexpr int NT = 4 * DV, LPR = DV / 4, RPP = NT / LPR, RPT = DK / RPP;
};

// chunk_base[n] = sum over m < n of ceil(len_m / C): the index of sequence n's first
// boundary state.  One thread: the batch sizes here are small.
__global__ void bwd_map_kernel(const int32_t *cu, int n_seqs, long long T, int C, int *base,
                               unsigned *err) {
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    int acc = 0;
    for (int n = 0; n < n_seqs; ++n) {
        long long s, e;
        seq_bounds(cu, n, T, err, s, e);
        base[n] = acc;
        acc += (int)((e - s + C - 1) / C);
    }
    base[n_seqs] = acc;
}

// Sum over the L lanes that hold one state row (L divides 32; rows are lane-aligned).
template <int L>
__device__ __forceinline__ float row_sum(float v) {
#pragma unroll
    for (int o = L / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Row sums of RPT rows held by the LPR lanes of a row group, written to out[row].  With 8 rows
// over 8 lanes the sums are formed by a transposing butterfly (7 shuffles for all 8 rows): after
// it, lane q of the group holds the sum of its row x = q, so each lane stores one value.
// Otherwise every row is reduced on its own (every lane ends with the sum; the first stores it).
template <int RPT, int LPR, int RPP>
__device__ __forceinline__ void store_row_sums(float (&v)[RPT], float *out, int rg, int lane) {
    if constexpr (RPT == 8 && LPR == 8) {
        const int q = lane & 7;
        float h4[4], h2[2];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const bool up = q & 4;
            const float send = up ? v[i] : v[i + 4];
            h4[i] = (up ? v[i + 4] : v[i]) + __shfl_xor_sync(0xffffffffu, send, 4);
        }
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const bool up = q & 2;
            const float send = up ? h4[i] : h4[i + 2];
            h2[i] = (up ? h4[i + 2] : h4[i]) + __shfl_xor_sync(0xffffffffu, send, 2);
        }
        const bool up = q & 1;
        const float send = up ? h2[0] : h2[1];
        const float tot = (up ? h2[1] : h2[0]) + __shfl_xor_sync(0xffffffffu, send, 1);
        out[rg * RPT + q] = tot;
    } else {
#pragma unroll
        for (int x = 0; x < RPT; ++x) {
            const float tot = row_sum<LPR>(v[x]);
            if (lane % LPR == 0) out[rg * RPT + x] = tot;
        }
    }
}

// Sum of the RPP partial column sums red[0..RPP)[col], as a tree.
template <int RPP, int DV>
__device__ __forceinline__ float col_sum(const float (&red)[RPP][DV], int col) {
    float t[RPP];
#pragma unroll
    for (int r = 0; r < RPP; ++r) t[r] = red[r][col];
#pragma unroll
    for (int w = RPP / 2; w > 0; w >>= 1)
#pragma unroll
        for (int r = 0; r < w; ++r) t[r] += t[r + w];
    return t[0];
}

// Two column-sum partials (y, z: columns c..c+3 of one row group, c = 4 (lane % 8)) summed over
// the four row groups of a warp by a transposing butterfly (6 shuffles): after it, each lane
// holds two of the warp's 64 sums, vector (lane & 16 ? z : y), columns c + (lane & 8 ? 2 : 0)
// and the next one, and stores them to out[vector][column].
__device__ __forceinline__ void warp_cols2(const float4 &y, const float4 &z, float (&out)[2][32], int lane) {
    const float v[8] = {y.x, y.y, y.z, y.w, z.x, z.y, z.z, z.w};
    float h4[4], h2[2];
    const bool up16 = lane & 16, up8 = lane & 8;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float send = up16 ? v[i] : v[i + 4];
        h4[i] = (up16 ? v[i + 4] : v[i]) + __shfl_xor_sync(0xffffffffu, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const float send = up8 ? h4[i] : h4[i + 2];
        h2[i] = (up8 ? h4[i + 2] : h4[i]) + __shfl_xor_sync(0xffffffffu, send, 8);
    }
    *reinterpret_cast<float2 *>(&out[up16 ? 1 : 0][(lane & 7) * 4 + (up8 ? 2 : 0)]) = make_float2(h2[0], h2[1]);
}

// N consecutive values of a staged row from p (aligned to N elements) as fp32, in one or two
// vector loads (the thread's rows of the state are consecutive: see BwdCfg).
template <int N, typename TA>
__device__ __forceinline__ void load_rows(const TA *p, float (&o)[N]) {
    if constexpr (sizeof(TA) == 2) {
        static_assert(N == 2 || N == 4 || N == 8, "whole 4-byte words of bf16 pairs");
        uint32_t w[N / 2];
        if constexpr (N == 8) {
            const uint4 u = *reinterpret_cast<const uint4 *>(p);
            w[0] = u.x; w[1] = u.y; w[2] = u.z; w[3] = u.w;
        } else if constexpr (N == 4) {
            const uint2 u = *reinterpret_cast<const uint2 *>(p);
            w[0] = u.x; w[1] = u.y;
        } else {
            w[0] = *reinterpret_cast<const uint32_t *>(p);
        }
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {   // bf16 pair: element 2i in the low half
            o[2 * i] = __uint_as_float(w[i] << 16);
            o[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    } else {
        static_assert(N % 2 == 0, "float2 or float4 loads");
        if constexpr (N % 4 == 0) {
#pragma unroll
            for (int i = 0; i < N; i += 4) {
                const float4 f = *reinterpret_cast<const float4 *>(p + i);
                o[i] = f.x; o[i + 1] = f.y; o[i + 2] = f.z; o[i + 3] = f.w;
            }
        } else {
            const float2 f = *reinterpret_cast<const float2 *>(p);
            o[0] = f.x; o[1] = f.y;
        }
    }
}

// ---- token inputs, staged one chunk at a time
// A chunk's inputs of one (v-head, slice) go to shared memory by asynchronous copies
// (cp.async, 16 bytes per copy for the rows, 4 for the gates) issued one chunk ahead, so a
// token step reads only shared memory and the global-load latency is paid once per chunk.
// q, k and v stay in the input dtype (converted on read); d_o, g and beta are fp32.
constexpr int kBwdMaxChunk = 64;

template <int DK, int DV, typename TA>
struct ChunkIn {
    alignas(16) TA q[kBwdMaxChunk][DK];
    alignas(16) TA k[kBwdMaxChunk][DK];
    alignas(16) TA v[kBwdMaxChunk][DV];
    alignas(16) float dout[kBwdMaxChunk][DV];
    alignas(16) float g[kBwdMaxChunk];
    alignas(16) float b[kBwdMaxChunk];
};

// Reductions of one token step, and the forward quantities of every token of the chunk that
// the reverse pass reuses: p = M^T k and w = beta (v - a p) (per column of the slice).
template <int DK, int DV>
struct BwdRed {
    alignas(16) float p[kBwdMaxChunk][DV];
    alignas(16) float w[kBwdMaxChunk][DV];
    alignas(16) float dp[DV];
    alignas(16) float red[BwdCfg<DK, DV>::RPP][DV];
    float wsum[BwdCfg<DK, DV>::NT / 32];
};

// The chunk-states kernel's pair steps: the p and w of the chunk's tokens, the two column sums
// of a pair per warp (pre-summed over the warp's row groups), and the pair dot products
// k_2j . k_2j+1 (qk is there for pair_dots, which can form q_2j . k_2j too).
template <int DK, int DV>
struct BwdRedPair {
    alignas(16) float p[kBwdMaxChunk][DV];
    alignas(16) float w[kBwdMaxChunk][DV];
    alignas(16) float cs[BwdCfg<DK, DV>::NT / 32][2][DV];
    float kk[kBwdMaxChunk / 2], qk[kBwdMaxChunk / 2];
};

// The gradient pass's: the pair's two column sums per warp (pre-summed over the warp's row
// groups), its two dp and dot products.
template <int DK, int DV>
struct BwdRedGm {
    alignas(16) float cs[BwdCfg<DK, DV>::NT / 32][2][DV];
    alignas(16) float dp2[2][DV];
    float kk[kBwdMaxChunk / 2], qk[kBwdMaxChunk / 2];
};

// NB chunk buffers: two (the next chunk's copies overlap this chunk) where one CTA runs per SM,
// one where three must fit.
template <int DK, int DV, typename TA, int NB = 2, typename RED = BwdRed<DK, DV>>
struct BwdSmem {
    ChunkIn<DK, DV, TA> in[NB];
    RED rd;
};
template <int DK, int DV, typename TA>
using BwdSmemPair = BwdSmem<DK, DV, TA, 2, BwdRedPair<DK, DV>>;
template <int DK, int DV, typename TA>
using BwdSmemGm = BwdSmem<DK, DV, TA, 2, BwdRedGm<DK, DV>>;

// Segments per sequence walked at once by bwd_kernel: segment k is chunks
// [k nch / BWD_SEG, (k + 1) nch / BWD_SEG).
constexpr int BWD_SEG = 3;
__host__ __device__ __forceinline__ long long seg_split(int k, long long nch) { return k * nch / BWD_SEG; }

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Issue the copies of tokens t0 .. t1-1 (t1 - t0 <= kBwdMaxChunk) into `ci`: k and v always,
// q and d_o when `with_q`; one commit group per call (possibly empty).  Row starts are 16-byte
// aligned: the entry points require 16-byte aligned bases and row strides that are multiples of
// 8 elements, and the slice's first column col0 is a multiple of 32.
template <int DK, int DV, typename TA, bool PAIRS = false>
__device__ __forceinline__ void stage_chunk(ChunkIn<DK, DV, TA> &ci, const BwdArgs &a, long long t0,
                                            long long t1, int h, int kh, int col0, bool with_q, int tid) {
    constexpr int NT = BwdCfg<DK, DV>::NT;
    constexpr int EK = 16 / (int)sizeof(TA);            // elements per 16-byte copy
    constexpr int PK = DK / EK, PV = DV / EK, PD = DV / 4;
    const int L = (int)(t1 - t0);
    const TA *kq = (const TA *)a.k, *qq = (const TA *)a.q, *vv = (const TA *)a.v;
    for (int i = tid; i < L * PK; i += NT) {
        const int r = i / PK, c = (i % PK) * EK;
        const long long row = (t0 + r) * a.ld_qk + (long long)kh * DK + c;
        cp_async16(&ci.k[r][c], kq + row);
        if (with_q) cp_async16(&ci.q[r][c], qq + row);
    }
    for (int i = tid; i < L * PV; i += NT) {
        const int r = i / PV, c = (i % PV) * EK;
        cp_async16(&ci.v[r][c], vv + (t0 + r) * a.ld_v + (long long)h * a.d.dv + col0 + c);
    }
    if (with_q)
        for (int i = tid; i < L * PD; i += NT) {
            const int r = i / PD, c = (i % PD) * 4;
            cp_async16(&ci.dout[r][c], a.d_o + (t0 + r) * (long long)a.d.hv * a.d.dv + (long long)h * a.d.dv + col0 + c);
        }
    for (int i = tid; i < 2 * L; i += NT) {
        const int r = i >> 1;
        if (i & 1) cp_async4(&ci.b[r], a.beta + (t0 + r) * a.d.hv + h);
        else cp_async4(&ci.g[r], a.g + (t0 + r) * a.d.hv + h);
    }
    cp_async_commit();
    // An odd chunk is walked in pairs with one neutral token after its last: k = q = v = d_o = 0,
    // g = 0 (a = 1) and beta = 0 leave the state, the gradient and every other token unchanged.
    // Row L is no copy's target; the barrier after the copies' wait publishes these stores.
    if (PAIRS && (L & 1)) {
        for (int i = tid; i < DK; i += NT) {
            ci.k[L][i] = from_f32<TA>(0.f);
            if (with_q) ci.q[L][i] = from_f32<TA>(0.f);
        }
        for (int i = tid; i < DV; i += NT) {
            ci.v[L][i] = from_f32<TA>(0.f);
            if (with_q) ci.dout[L][i] = 0.f;
        }
        if (tid == 0) { ci.g[L] = 0.f; ci.b[L] = 0.f; }
    }
}

// The dot products the pair steps need, for the pairs (2j, 2j+1) of a staged chunk of L tokens:
// kk[j] = k_2j . k_2j+1 and, with q staged, qk[j] = q_2j . k_2j.  Four threads per product (a
// quarter of the dk terms each, then two shuffles); the caller's next barrier publishes them.
template <int DK, int DV, typename TA, typename RED>
__device__ __forceinline__ void pair_dots(const ChunkIn<DK, DV, TA> &ci, RED &rd, int L, bool with_q, int tid) {
    constexpr int NT = BwdCfg<DK, DV>::NT, Q = DK / 4;
    static_assert(NT % 4 == 0 && (2 * kBwdMaxChunk / 2) * 4 % NT == 0, "whole groups of four lanes");
    const int np = (L + 1) >> 1;
#pragma unroll
    for (int u = 0; u < (2 * kBwdMaxChunk / 2) * 4 / NT; ++u) {
        const int task = tid + u * NT, prod = task >> 2, part = task & 3;
        const bool isq = prod >= kBwdMaxChunk / 2;
        const int j = isq ? prod - kBwdMaxChunk / 2 : prod;
        float acc = 0.f;
        if (j < np && (!isq || with_q)) {
            const TA *x = isq ? ci.q[2 * j] : ci.k[2 * j];
            const TA *y = isq ? ci.k[2 * j] : ci.k[2 * j + 1];
#pragma unroll 8
            for (int i = part * Q; i < part * Q + Q; ++i) acc = fmaf(to_f32(x[i]), to_f32(y[i]), acc);
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        acc += __shfl_xor_sync(0xffffffffu, acc, 2);
        if (part == 0 && j < np) (isq ? rd.qk : rd.kk)[j] = acc;
    }
}


// One row's float4 of the state through one token: M <- a M + k w^T (the replay and the reverse
// pass's reconstruction use this same expression).
__device__ __forceinline__ void state_update(float4 &m, float a, float k, const float4 &w) {
    m.x = a * m.x + k * w.x; m.y = a * m.y + k * w.y;
    m.z = a * m.z + k * w.z; m.w = a * m.w + k * w.w;
}

// The forward step of the token pair (tt, tt + 1) of a staged chunk (tt even) on M in registers:
// p = M^T k and w = beta (v - a p) of both tokens (kept in rd at rows tt and tt + 1), and
// M <- a M + k w^T twice.  The second token's p follows from the same pass over M:
// p_1 = (a_0 M + k_0 w_0^T)^T k_1 = a_0 M^T k_1 + (k_0 . k_1) w_0.  Two block barriers per pair.
// With `pwo` (token tt's p row of this slice in the per-token p/w rows; its w row is dvh floats
// on, the next token's rows `ts` floats on) warp 0 also writes both tokens' p and w there, the
// second only when `has1` (not the neutral token of an odd chunk).
template <int DK, int DV, typename TA, bool CONSEC = true>
__device__ __forceinline__ void fwd_pair(float4 (&m)[BwdCfg<DK, DV>::RPT], BwdRedPair<DK, DV> &rd,
                                         const ChunkIn<DK, DV, TA> &in, int tt, int warp, int lane, int rg,
                                         int c4, float *pwo = nullptr, long long ts = 0, int dvh = 0,
                                         bool has1 = false) {
    using C = BwdCfg<DK, DV>;
    float kr0[C::RPT], kr1[C::RPT];
    if constexpr (CONSEC) {   // rows rg*RPT + x
        load_rows<C::RPT>(in.k[tt] + rg * C::RPT, kr0);
        load_rows<C::RPT>(in.k[tt + 1] + rg * C::RPT, kr1);
    } else {                  // rows rg + x*RPP
#pragma unroll
        for (int x = 0; x < C::RPT; ++x) {
            kr0[x] = to_f32(in.k[tt][rg + x * C::RPP]);
            kr1[x] = to_f32(in.k[tt + 1][rg + x * C::RPP]);
        }
    }
    float4 pp0 = make_float4(0.f, 0.f, 0.f, 0.f), pp1 = pp0;
#pragma unroll
    for (int x = 0; x < C::RPT; ++x) {
        pp0.x += m[x].x * kr0[x]; pp0.y += m[x].y * kr0[x]; pp0.z += m[x].z * kr0[x]; pp0.w += m[x].w * kr0[x];
        pp1.x += m[x].x * kr1[x]; pp1.y += m[x].y * kr1[x]; pp1.z += m[x].z * kr1[x]; pp1.w += m[x].w * kr1[x];
    }
    warp_cols2(pp0, pp1, rd.cs[warp], lane);
    __syncthreads();
    const float a0 = in.g[tt], a1 = in.g[tt + 1];       // a = exp(g), converted by the caller
    if (warp == 0) {
        float x0 = 0.f, x1 = 0.f;
#pragma unroll
        for (int wi = 0; wi < C::NT / 32; ++wi) { x0 += rd.cs[wi][0][lane]; x1 += rd.cs[wi][1][lane]; }
        const float p0 = x0;
        const float w0 = in.b[tt] * (to_f32(in.v[tt][lane]) - a0 * p0);
        const float p1 = a0 * x1 + rd.kk[tt >> 1] * w0;
        rd.p[tt][lane] = p0;
        rd.w[tt][lane] = w0;
        const float w1 = in.b[tt + 1] * (to_f32(in.v[tt + 1][lane]) - a1 * p1);
        rd.p[tt + 1][lane] = p1;
        rd.w[tt + 1][lane] = w1;
        if (pwo) {
            pwo[lane] = p0;
            pwo[dvh + lane] = w0;
            if (has1) {
                pwo[ts + lane] = p1;
                pwo[ts + dvh + lane] = w1;
            }
        }
    }
    __syncthreads();
    const float4 w0 = *reinterpret_cast<const float4 *>(&rd.w[tt][c4]);
    const float4 w1 = *reinterpret_cast<const float4 *>(&rd.w[tt + 1][c4]);
#pragma unroll
    for (int x = 0; x < C::RPT; ++x) {
        state_update(m[x], a0, kr0[x], w0);
        state_update(m[x], a1, kr1[x], w1);
    }
}

// The forward step of token tt of a staged chunk on M in registers: p = M^T k (column sums),
// r = v - a p, w = beta r (kept in rd at row tt), and, when `update`, M <- a M + k w^T.  The
// chunk's g row holds a = exp(g) here (the walk converts it once per chunk).
// Two block barriers.
template <int DK, int DV, typename TA>
__device__ __forceinline__ void fwd_token(float4 (&m)[BwdCfg<DK, DV>::RPT], BwdRed<DK, DV> &rd,
                                          const ChunkIn<DK, DV, TA> &in, int tt, int tid, int rg, int c4,
                                          bool update) {
    using C = BwdCfg<DK, DV>;
    float kr[C::RPT];
    load_rows<C::RPT>(in.k[tt] + rg * C::RPT, kr);
    float4 pp = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int x = 0; x < C::RPT; ++x) {
        pp.x += m[x].x * kr[x]; pp.y += m[x].y * kr[x]; pp.z += m[x].z * kr[x]; pp.w += m[x].w * kr[x];
    }
    *reinterpret_cast<float4 *>(&rd.red[rg][c4]) = pp;
    __syncthreads();
    const float av = in.g[tt];                           // a = exp(g), staged by the caller
    if (tid < DV) {
        const float p = col_sum<C::RPP, DV>(rd.red, tid);
        rd.p[tt][tid] = p;
        rd.w[tt][tid] = in.b[tt] * (to_f32(in.v[tt][tid]) - av * p);
    }
    __syncthreads();
    if (!update) return;
    const float4 w4 = *reinterpret_cast<const float4 *>(&rd.w[tt][c4]);
#pragma unroll
    for (int x = 0; x < C::RPT; ++x) state_update(m[x], av, kr[x], w4);
}

// (This kernel keeps the interleaved row mapping, rows rg + x*RPP per thread: with consecutive
// rows and vector k loads it measured slower, 2.45 against 2.25 ms at 8,192 tokens.)
template <int DK, int DV, typename TA>
__global__ void __launch_bounds__(4 * DV) bwd_states_kernel(BwdArgs a) {
    using C = BwdCfg<DK, DV>;
    extern __shared__ __align__(16) unsigned char smraw[];
    BwdSmemPair<DK, DV, TA> &sm = *reinterpret_cast<BwdSmemPair<DK, DV, TA> *>(smraw);
    const Dims &d = a.d;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, h = blockIdx.x, n = blockIdx.y, kh = h / d.grp;
    const int col0 = blockIdx.z * DV;                   // this CTA's slice of the state columns
    const int rg = tid / C::LPR, c4s = (tid % C::LPR) * 4, c4 = c4s + col0;   // (c4: column in the head)
    long long s, e;
    seq_bounds(a.cu_seqlens, n, a.T, a.err, s, e);
    const int slot = slot_of(a.state_idx, n, d.n_slots, a.err);
    if (slot < 0 || s >= e) return;                      // padding lane / empty: no chunks
    const int Cc = d.chunk;
    const int DVH = d.dv;                               // columns of the whole head
    float4 m[C::RPT];
#pragma unroll
    for (int x = 0; x < C::RPT; ++x) {
        m[x] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (a.state_in)
            m[x] = *reinterpret_cast<const float4 *>(a.state_in + ((long long)slot * d.hv + h) * DK * DVH +
                                                     (long long)(rg + x * C::RPP) * DVH + c4);
    }
    const long long b0 = a.chunk_base[n];
    const long long nch = (e - s + Cc - 1) / Cc;
    auto bounds = [&](long long c, long long &t0, long long &t1) {
        t0 = s + c * Cc;
        t1 = t0 + Cc < e ? t0 + Cc : e;
    };
    long long t0, t1;
    bounds(0, t0, t1);
    stage_chunk<DK, DV, TA, true>(sm.in[0], a, t0, t1, h, kh, col0, false, tid);
    for (long long c = 0; c < nch; ++c) {
        __syncthreads();                                 // every read of buffer (c + 1) & 1 is done
        if (c + 1 < nch) {
            long long u0, u1;
            bounds(c + 1, u0, u1);
            stage_chunk<DK, DV, TA, true>(sm.in[(c + 1) & 1], a, u0, u1, h, kh, col0, false, tid);
            cp_async_wait<1>();                          // this thread's copies of chunk c landed
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();                                 // ... and everyone's
        bounds(c, t0, t1);
        float *B = a.bnd + ((b0 + c) * d.hv + h) * DK * DVH;
#pragma unroll
        for (int x = 0; x < C::RPT; ++x)
            *reinterpret_cast<float4 *>(B + (long long)(rg + x * C::RPP) * DVH + c4) = m[x];
        const ChunkIn<DK, DV, TA> &in = sm.in[c & 1];
        const int L = (int)(t1 - t0);
        pair_dots<DK, DV, TA>(in, sm.rd, L, false, tid);
        // the decays a = exp(g) once, in place of g (the neutral token's g = 0 gives a = 1)
        for (int r = tid; r < ((L + 1) & ~1); r += C::NT) sm.in[c & 1].g[r] = expf(sm.in[c & 1].g[r]);
        __syncthreads();
        const long long ts = 2LL * d.hv * DVH;           // per-token p/w rows: one token's stride
        float *pw0 = a.pw ? a.pw + (t0 * d.hv + h) * 2LL * DVH + col0 : nullptr;
        for (int tt = 0; tt < L; tt += 2)
            fwd_pair<DK, DV, TA, false>(m, sm.rd, in, tt, warp, lane, rg, c4s, pw0 ? pw0 + tt * ts : nullptr, ts,
                                        DVH, tt + 1 < L);
    }
}

// dL/dS entering each segment's last chunk boundary, for the segments of bwd_kernel that do not
// end at the sequence end: the gradient alone carried back from d_state_out over chunks
// [nch / BWD_SEG, nch), and kept at every segment boundary it passes.  Per token (reverse),
// with G = dL/dM after the token: G <- a (G + q do^T) - a beta k (k^T (G + q do^T)), which needs
// no forward state.  One CTA per (sequence, v-head, slice); the tokens go in pairs (t, t-1), one
// pass over X = G + q_t do_t^T giving both X^T k_t and X^T k_(t-1), which with the pair's dot
// products fixes the second token's column sums too: two barriers per pair.
template <int DK, int DV, typename TA>
__global__ void __launch_bounds__(4 * DV) bwd_gm_kernel(BwdArgs a) {
    using C = BwdCfg<DK, DV>;
    constexpr int NW = C::NT / 32;
    static_assert(DV == 32, "the per-column steps run on warp 0, one column per lane");
    extern __shared__ __align__(16) unsigned char smraw[];
    BwdSmemGm<DK, DV, TA> &sm = *reinterpret_cast<BwdSmemGm<DK, DV, TA> *>(smraw);
    BwdRedGm<DK, DV> &rd = sm.rd;
    const Dims &d = a.d;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int h = blockIdx.x, n = blockIdx.y, kh = h / d.grp;
    const int col0 = blockIdx.z * DV;
    const int rg = tid / C::LPR, c4s = (tid % C::LPR) * 4, c4 = c4s + col0;
    long long s, e;
    seq_bounds(a.cu_seqlens, n, a.T, nullptr, s, e);
    const int slot = slot_of(a.state_idx, n, d.n_slots, nullptr);
    const int Cc = d.chunk, DVH = d.dv;
    const long long nch = (e - s + Cc - 1) / Cc;
    long long cs = 0;                                    // the first split that has a segment before it
    for (int k = 1; k < BWD_SEG && cs == 0; ++k) cs = seg_split(k, nch);
    if (slot < 0 || cs == 0) return;                     // no earlier segment to feed
    float4 gm[C::RPT];
#pragma unroll
    for (int x = 0; x < C::RPT; ++x) {
        gm[x] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (a.d_state_out)
            gm[x] = *reinterpret_cast<const float4 *>(a.d_state_out + ((long long)slot * d.hv + h) * DK * DVH +
                                                      (long long)(rg * C::RPT + x) * DVH + c4);
    }
    auto bounds = [&](long long c, long long &t0, long long &t1) {
        t0 = s + c * Cc;
        t1 = t0 + Cc < e ? t0 + Cc : e;
    };
    {
        long long u0, u1;
        bounds(nch - 1, u0, u1);
        stage_chunk<DK, DV, TA, true>(sm.in[(nch - 1) & 1], a, u0, u1, h, kh, col0, true, tid);
    }
    for (long long c = nch - 1; c >= cs; --c) {
        long long t0, t1;
        bounds(c, t0, t1);
        __syncthreads();                                 // every read of buffer (c - 1) & 1 is done
        if (c > cs) {
            long long u0, u1;
            bounds(c - 1, u0, u1);
            stage_chunk<DK, DV, TA, true>(sm.in[(c - 1) & 1], a, u0, u1, h, kh, col0, true, tid);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const ChunkIn<DK, DV, TA> &in = sm.in[c & 1];
        const int L = (int)(t1 - t0);
        pair_dots<DK, DV, TA>(in, rd, L, true, tid);
        // the decays a = exp(g) once, in place of g (the neutral token's g = 0 gives a = 1)
        for (int r = tid; r < ((L + 1) & ~1); r += C::NT) sm.in[c & 1].g[r] = expf(sm.in[c & 1].g[r]);
        __syncthreads();
        for (int tt = ((L + 1) & ~1) - 1; tt > 0; tt -= 2) {   // the pairs (tt, tt - 1), tt odd
            const float a1 = in.g[tt], b1 = in.b[tt], a0 = in.g[tt - 1], b0 = in.b[tt - 1];   // (a = exp(g))
            const float4 do1 = *reinterpret_cast<const float4 *>(&in.dout[tt][c4s]);
            const float4 do0 = *reinterpret_cast<const float4 *>(&in.dout[tt - 1][c4s]);
            float kr1[C::RPT], kr0[C::RPT], qv[C::RPT];
            load_rows<C::RPT>(in.k[tt] + rg * C::RPT, kr1);
            load_rows<C::RPT>(in.k[tt - 1] + rg * C::RPT, kr0);
            load_rows<C::RPT>(in.q[tt] + rg * C::RPT, qv);
            float4 yp = make_float4(0.f, 0.f, 0.f, 0.f), zp = yp;
#pragma unroll
            for (int x = 0; x < C::RPT; ++x) {   // X = G + q do^T of token tt; X^T k_tt, X^T k_(tt-1)
                const float qr = qv[x];
                gm[x].x += qr * do1.x; gm[x].y += qr * do1.y; gm[x].z += qr * do1.z; gm[x].w += qr * do1.w;
                yp.x += gm[x].x * kr1[x]; yp.y += gm[x].y * kr1[x]; yp.z += gm[x].z * kr1[x]; yp.w += gm[x].w * kr1[x];
                zp.x += gm[x].x * kr0[x]; zp.y += gm[x].y * kr0[x]; zp.z += gm[x].z * kr0[x]; zp.w += gm[x].w * kr0[x];
            }
            warp_cols2(yp, zp, rd.cs[warp], lane);
            __syncthreads();
            if (warp == 0) {   // dp of both tokens: dw_(tt-1) = a X^T k_(tt-1) + (k_tt . k_(tt-1)) dp_tt + (q . k)_(tt-1) do
                float x1 = 0.f, x0 = 0.f;
#pragma unroll
                for (int wi = 0; wi < NW; ++wi) { x1 += rd.cs[wi][0][lane]; x0 += rd.cs[wi][1][lane]; }
                const float dp1 = -a1 * b1 * x1;
                const float dw0 = a1 * x0 + rd.kk[tt >> 1] * dp1 + rd.qk[tt >> 1] * in.dout[tt - 1][lane];
                rd.dp2[0][lane] = dp1;
                rd.dp2[1][lane] = -a0 * b0 * dw0;
            }
            __syncthreads();
            const float4 dp1 = *reinterpret_cast<const float4 *>(&rd.dp2[0][c4s]);
            const float4 dp0 = *reinterpret_cast<const float4 *>(&rd.dp2[1][c4s]);
            load_rows<C::RPT>(in.q[tt - 1] + rg * C::RPT, qv);
#pragma unroll
            for (int x = 0; x < C::RPT; ++x) {   // G <- a X + k dp^T, twice, with token tt-1's q do^T between
                const float qr = qv[x];
                gm[x].x = a1 * gm[x].x + kr1[x] * dp1.x + qr * do0.x;
                gm[x].y = a1 * gm[x].y + kr1[x] * dp1.y + qr * do0.y;
                gm[x].z = a1 * gm[x].z + kr1[x] * dp1.z + qr * do0.z;
                gm[x].w = a1 * gm[x].w + kr1[x] * dp1.w + qr * do0.w;
                gm[x].x = a0 * gm[x].x + kr0[x] * dp0.x; gm[x].y = a0 * gm[x].y + kr0[x] * dp0.y;
                gm[x].z = a0 * gm[x].z + kr0[x] * dp0.z; gm[x].w = a0 * gm[x].w + kr0[x] * dp0.w;
            }
        }
        // the gradient entering chunk c starts every segment that ends there
        for (int k = 1; k < BWD_SEG; ++k) {
            if (seg_split(k, nch) != c) continue;
            float *D = a.gsplit + (((long long)n * d.hv + h) * (BWD_SEG - 1) + (k - 1)) * DK * DVH;
#pragma unroll
            for (int x = 0; x < C::RPT; ++x)
                *reinterpret_cast<float4 *>(D + (long long)(rg * C::RPT + x) * DVH + c4) = gm[x];
        }
    }
}

template <int DK, int DV, typename TA>
__global__ void __launch_bounds__(4 * DV, 3) bwd_kernel(BwdArgs a) {
    using C = BwdCfg<DK, DV>;
    constexpr int NW = C::NT / 32;
    static_assert(DV == 32, "the per-column steps run on warp 0, one column per lane");
    extern __shared__ __align__(16) unsigned char smraw[];
    BwdSmem<DK, DV, TA, 1> &sm = *reinterpret_cast<BwdSmem<DK, DV, TA, 1> *>(smraw);
    BwdRed<DK, DV> &rd = sm.rd;
    const Dims &d = a.d;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int h = blockIdx.x, n = blockIdx.y, kh = h / d.grp;
    const int NS = gridDim.z / BWD_SEG, sl = blockIdx.z % NS, seg = blockIdx.z / NS;
    const int col0 = sl * DV;                            // this CTA's slice of the columns
    const int rg = tid / C::LPR, c4s = (tid % C::LPR) * 4, c4 = c4s + col0;
    long long s, e;
    seq_bounds(a.cu_seqlens, n, a.T, a.err, s, e);
    const int slot = slot_of(a.state_idx, n, d.n_slots, a.err);
    const int DVH = d.dv;
    const long long HVDV = (long long)d.hv * DVH;
    auto part = [&](long long t) { return (t * d.hv + h) * NS + sl; };   // index of this slice's parts
    if (slot < 0) {                                      // padding lane: zero gradients (last segment)
        if (seg != BWD_SEG - 1) return;
        for (long long t = s; t < e; ++t) {
            for (int i = tid; i < DK; i += C::NT) {
                a.pq[part(t) * DK + i] = 0.f;
                a.pk[part(t) * DK + i] = 0.f;
            }
            for (int j = tid; j < DV; j += C::NT) a.dv[t * HVDV + (long long)h * DVH + col0 + j] = 0.f;
            if (tid == 0) { a.pda[part(t)] = 0.f; a.pda2[part(t)] = 0.f; a.pdb[part(t)] = 0.f; }
        }
        return;
    }
    const int Cc = d.chunk;
    const long long nch = (e - s + Cc - 1) / Cc;
    // The sequence's chunks are split in BWD_SEG segments walked at the same time.  The last
    // starts from d_state_out; every other one from dL/dS entering the next segment's first
    // chunk, which bwd_gm_kernel has carried back beforehand.
    const bool last = seg == BWD_SEG - 1;
    const long long c_lo = seg_split(seg, nch), c_hi = seg_split(seg + 1, nch);
    if (c_lo >= c_hi && !(last && nch == 0)) return;     // (an empty sequence: the last segment only)
    const float *g_init = last ? a.d_state_out : a.gsplit;
    const long long g_off = last ? ((long long)slot * d.hv + h) * DK * DVH
                                 : (((long long)n * d.hv + h) * (BWD_SEG - 1) + seg) * DK * DVH;
    float4 gm[C::RPT];
#pragma unroll
    for (int x = 0; x < C::RPT; ++x) {
        gm[x] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (g_init)
            gm[x] = *reinterpret_cast<const float4 *>(g_init + g_off + (long long)(rg * C::RPT + x) * DVH + c4);
    }
    // this CTA's scratch: the slice of the state before each even token of one chunk
    float *scr = a.scratch + ((((long long)n * d.hv + h) * NS + sl) * BWD_SEG + seg) * (long long)((Cc + 1) / 2) * DK * DV;
    const long long b0 = a.chunk_base[n];
    auto bounds = [&](long long c, long long &t0, long long &t1) {
        t0 = s + c * Cc;
        t1 = t0 + Cc < e ? t0 + Cc : e;
    };
    for (long long c = c_hi - 1; c >= c_lo; --c) {
        long long t0, t1;
        bounds(c, t0, t1);
        float4 m[C::RPT];
        {
            const float *B = a.bnd + ((b0 + c) * d.hv + h) * DK * DVH;
#pragma unroll
            for (int x = 0; x < C::RPT; ++x)
                m[x] = *reinterpret_cast<const float4 *>(B + (long long)(rg * C::RPT + x) * DVH + c4);
        }
        // one chunk buffer (three CTAs per SM): the previous chunk's reads are done, then this
        // chunk's copies
        __syncthreads();
        stage_chunk<DK, DV, TA>(sm.in[0], a, t0, t1, h, kh, col0, true, tid);
        if (a.pw) {   // the retained p and w of the chunk's tokens, this slice's columns
            constexpr int PR = DV / 4;                   // 16-byte copies per row
            for (int i = tid; i < (int)(t1 - t0) * 2 * PR; i += C::NT) {
                const int r = i / (2 * PR), half = (i / PR) & 1, c = (i % PR) * 4;
                cp_async16((half ? rd.w[r] : rd.p[r]) + c,
                           a.pw + ((t0 + r) * d.hv + h) * 2LL * DVH + (long long)half * DVH + col0 + c);
            }
            cp_async_commit();
        }
        cp_async_wait<0>();
        __syncthreads();
        // the decays a = exp(g) of the chunk's tokens, once, in place of g
        for (int r = tid; r < (int)(t1 - t0); r += C::NT) sm.in[0].g[r] = expf(sm.in[0].g[r]);
        __syncthreads();
        const ChunkIn<DK, DV, TA> &in = sm.in[0];   // (in.g holds a = exp(g) from here)
        // forward through the chunk, keeping the state before every even token (each thread
        // reads back only what it wrote) and every token's p and w.  With the p and w retained
        // by gdn_chunk_states each thread carries its rows alone: no sums, no barriers (the
        // update there, with the same w).
        if (a.pw) {
            for (int tt = 0; tt < (int)(t1 - t0); ++tt) {
                if ((tt & 1) == 0) {
                    float *Sc = scr + (tt >> 1) * DK * DV;
#pragma unroll
                    for (int x = 0; x < C::RPT; ++x)
                        *reinterpret_cast<float4 *>(Sc + (long long)(rg * C::RPT + x) * DV + c4s) = m[x];
                }
                float kr[C::RPT];
                load_rows<C::RPT>(in.k[tt] + rg * C::RPT, kr);
                const float av = in.g[tt];
                const float4 w4 = *reinterpret_cast<const float4 *>(&rd.w[tt][c4s]);
#pragma unroll
                for (int x = 0; x < C::RPT; ++x) state_update(m[x], av, kr[x], w4);
            }
        } else {
            for (long long t = t0; t < t1; ++t) {
                const int tt = (int)(t - t0);
                if ((tt & 1) == 0) {
                    float *Sc = scr + (tt >> 1) * DK * DV;
#pragma unroll
                    for (int x = 0; x < C::RPT; ++x)
                        *reinterpret_cast<float4 *>(Sc + (long long)(rg * C::RPT + x) * DV + c4s) = m[x];
                }
                fwd_token<DK, DV, TA>(m, rd, in, tt, tid, rg, c4s, true);
            }
        }
        // The tokens in reverse.  A step takes the state after its token in `mc` (the replay
        // ends with the state after the chunk's last token), which is the M' of dq = M' do, and
        // the stored state before the even token of its pair in `ms`.  An odd token turns mc into
        // the state before it (the stored one carried over the even token, with its kept w); an
        // even token's state before it is ms itself, and mc, no longer needed after dq, takes the
        // next pair's stored state.  So after each pair the two arrays have swapped roles: the
        // loop takes two pairs per turn with the arrays named in turn, and no state is copied.
        float4 mn[C::RPT];
        const int L = (int)(t1 - t0);
        {
            const float *Sc = scr + ((L - 1) >> 1) * DK * DV;
#pragma unroll
            for (int x = 0; x < C::RPT; ++x)
                mn[x] = *reinterpret_cast<const float4 *>(Sc + (long long)(rg * C::RPT + x) * DV + c4s);
        }
        auto rstep = [&](auto odd, float4 (&mc)[C::RPT], float4 (&ms)[C::RPT], int tt) {
            constexpr bool ODD = decltype(odd)::value;
            const long long t = t0 + tt;
            const float4 do4 = *reinterpret_cast<const float4 *>(&in.dout[tt][c4s]);
            float dqp[C::RPT];
#pragma unroll
            for (int x = 0; x < C::RPT; ++x)                 // dq = M' do, M' the state after the token
                dqp[x] = mc[x].x * do4.x + mc[x].y * do4.y + mc[x].z * do4.z + mc[x].w * do4.w;
            if constexpr (ODD) {                             // mc <- the state before the token
                const float a0 = in.g[tt - 1];
                const float4 w0 = *reinterpret_cast<const float4 *>(&rd.w[tt - 1][c4s]);
                float k0[C::RPT];
                load_rows<C::RPT>(in.k[tt - 1] + rg * C::RPT, k0);
#pragma unroll
                for (int x = 0; x < C::RPT; ++x) {
                    mc[x] = ms[x];
                    state_update(mc[x], a0, k0[x], w0);
                }
            } else if (tt >= 2) {                            // mc <- the next pair's stored state
                const float *Sc = scr + ((tt >> 1) - 1) * DK * DV;
#pragma unroll
                for (int x = 0; x < C::RPT; ++x)
                    mc[x] = *reinterpret_cast<const float4 *>(Sc + (long long)(rg * C::RPT + x) * DV + c4s);
            }
            float4 (&m)[C::RPT] = *[&]() -> float4 (*)[C::RPT] {   // the state before the token
                if constexpr (ODD) return &mc;
                else return &ms;
            }();
            const float av = in.g[tt], bv = in.b[tt];
            const float4 w4 = *reinterpret_cast<const float4 *>(&rd.w[tt][c4s]);
            float4 dwp = make_float4(0.f, 0.f, 0.f, 0.f);
            float dap = 0.f;
            float kr[C::RPT], qv[C::RPT];
            load_rows<C::RPT>(in.k[tt] + rg * C::RPT, kr);
            load_rows<C::RPT>(in.q[tt] + rg * C::RPT, qv);
#pragma unroll
            for (int x = 0; x < C::RPT; ++x) {
                const float qr = qv[x];
                gm[x].x += qr * do4.x; gm[x].y += qr * do4.y; gm[x].z += qr * do4.z; gm[x].w += qr * do4.w;
                dwp.x += gm[x].x * kr[x]; dwp.y += gm[x].y * kr[x]; dwp.z += gm[x].z * kr[x]; dwp.w += gm[x].w * kr[x];
                dap += gm[x].x * m[x].x + gm[x].y * m[x].y + gm[x].z * m[x].z + gm[x].w * m[x].w;
            }
            *reinterpret_cast<float4 *>(&rd.red[rg][c4s]) = dwp;
            store_row_sums<C::RPT, C::LPR, C::RPP>(dqp, a.pq + part(t) * DK, rg, lane);
            dap = warp_sum(dap);
            if (lane == 0) rd.wsum[warp] = dap;
            __syncthreads();                             // (C)
            if (warp == 0) {   // dw = GM^T k (column sums), dv, dp; this slice's parts of dg, dbeta
                const float dw = col_sum<C::RPP, DV>(rd.red, lane);
                a.dv[t * HVDV + (long long)h * DVH + col0 + lane] = bv * dw;
                rd.dp[lane] = -av * bv * dw;
                const float pl = rd.p[tt][lane];
                const float db = warp_sum(dw * (to_f32(in.v[tt][lane]) - av * pl));   // dw . (v - a p)
                const float da2 = warp_sum(dw * pl);
                if (lane == 0) {
                    float da = 0.f;
#pragma unroll
                    for (int wi = 0; wi < NW; ++wi) da += rd.wsum[wi];
                    a.pda[part(t)] = da;
                    a.pda2[part(t)] = da2;
                    a.pdb[part(t)] = db;
                }
            }
            __syncthreads();                             // (D)
            const float4 dp4 = *reinterpret_cast<const float4 *>(&rd.dp[c4s]);
            float dkp[C::RPT];
#pragma unroll
            for (int x = 0; x < C::RPT; ++x) {   // dk = GM w + M dp, then GM <- a GM + k dp^T
                dkp[x] = gm[x].x * w4.x + gm[x].y * w4.y + gm[x].z * w4.z + gm[x].w * w4.w +
                         m[x].x * dp4.x + m[x].y * dp4.y + m[x].z * dp4.z + m[x].w * dp4.w;
                gm[x].x = av * gm[x].x + kr[x] * dp4.x; gm[x].y = av * gm[x].y + kr[x] * dp4.y;
                gm[x].z = av * gm[x].z + kr[x] * dp4.z; gm[x].w = av * gm[x].w + kr[x] * dp4.w;
            }
            store_row_sums<C::RPT, C::LPR, C::RPP>(dkp, a.pk + part(t) * DK, rg, lane);
        };
        using Odd = std::true_type;
        using Even = std::false_type;
        int tt = L - 1;
        if ((tt & 1) == 0) {   // an odd-length chunk: its last token is even and has no partner
            rstep(Even{}, m, mn, tt--);
#pragma unroll
            for (int x = 0; x < C::RPT; ++x) {   // (once per such chunk: the roles back in place)
                const float4 tmp = m[x];
                m[x] = mn[x];
                mn[x] = tmp;
            }
        }
        for (; tt >= 3; tt -= 4) {
            rstep(Odd{}, m, mn, tt);
            rstep(Even{}, m, mn, tt - 1);
            rstep(Odd{}, mn, m, tt - 2);
            rstep(Even{}, mn, m, tt - 3);
        }
        if (tt == 1) {
            rstep(Odd{}, m, mn, 1);
            rstep(Even{}, m, mn, 0);
        }
    }
    if (a.d_state_in && c_lo == 0) {                    // the segment that ends at the first chunk
        // (the first non-empty one; for an empty sequence, the last)
        float *D = a.d_state_in + ((long long)slot * d.hv + h) * DK * DVH;
#pragma unroll
        for (int x = 0; x < C::RPT; ++x)
            *reinterpret_cast<float4 *>(D + (long long)(rg * C::RPT + x) * DVH + c4) = gm[x];
    }
}

// dq, dk of each q/k head: the sum over its v-heads and their column slices; dg and dbeta of
// each v-head from its slices' parts (dg = a (<GM, M> - beta dw . p)).
__global__ void bwd_group_sum_kernel(BwdArgs a, int NS) {
    const Dims &d = a.d;
    // dq, dk: a CTA per token row at a time, a thread per four consecutive columns (float4 loads
    // of the parts; float4 stores when the row stride allows them)
    const int row4 = d.hk * d.dk / 4;
    const bool vec = (a.ld_dqk & 3) == 0;
    for (long long t = blockIdx.x; t < a.T; t += gridDim.x) {
        for (int j4 = threadIdx.x; j4 < row4; j4 += blockDim.x) {
            const int kh = (4 * j4) / d.dk, i = (4 * j4) % d.dk;
            float4 sq = make_float4(0.f, 0.f, 0.f, 0.f), sk = sq;
            for (int gi = 0; gi < d.grp; ++gi)
                for (int sl = 0; sl < NS; ++sl) {
                    const long long src = ((t * d.hv + kh * d.grp + gi) * NS + sl) * d.dk + i;
                    const float4 q4 = *reinterpret_cast<const float4 *>(a.pq + src);
                    const float4 k4 = *reinterpret_cast<const float4 *>(a.pk + src);
                    sq.x += q4.x; sq.y += q4.y; sq.z += q4.z; sq.w += q4.w;
                    sk.x += k4.x; sk.y += k4.y; sk.z += k4.z; sk.w += k4.w;
                }
            float *dq = a.dq + t * a.ld_dqk + (long long)kh * d.dk + i;
            float *dk = a.dk + t * a.ld_dqk + (long long)kh * d.dk + i;
            if (vec) {
                *reinterpret_cast<float4 *>(dq) = sq;
                *reinterpret_cast<float4 *>(dk) = sk;
            } else {
                dq[0] = sq.x; dq[1] = sq.y; dq[2] = sq.z; dq[3] = sq.w;
                dk[0] = sk.x; dk[1] = sk.y; dk[2] = sk.z; dk[3] = sk.w;
            }
        }
    }
    const long long th = a.T * d.hv;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < th;
         e += (long long)gridDim.x * blockDim.x) {
        float da = 0.f, da2 = 0.f, db = 0.f;
        for (int sl = 0; sl < NS; ++sl) {
            da += a.pda[e * NS + sl];
            da2 += a.pda2[e * NS + sl];
            db += a.pdb[e * NS + sl];
        }
        const float av = expf(a.g[e]), bv = a.beta[e];
        a.dg[e] = av * (da - bv * da2);
        a.dbeta[e] = db;
    }
}

template <int D, typename TA>
cudaError_t launch_bwd_t(const BwdArgs &a, bool states_only, cudaStream_t s) {
    constexpr int NS = D / BWD_DVS;                      // column slices per head
    const dim3 grid(a.d.hv, a.n_seqs, NS);
    bwd_map_kernel<<<1, 32, 0, s>>>(a.cu_seqlens, a.n_seqs, a.T, a.d.chunk, a.chunk_base, a.err);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    constexpr int smem = (int)sizeof(BwdSmemPair<D, BWD_DVS, TA>);
    constexpr int smem1 = (int)sizeof(BwdSmem<D, BWD_DVS, TA, 1>);
    if (states_only) {
        auto kern = bwd_states_kernel<D, BWD_DVS, TA>;
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem)) != cudaSuccess)
            return e;
        kern<<<grid, 4 * BWD_DVS, smem, s>>>(a);
        return cudaGetLastError();
    }
    auto gk = bwd_gm_kernel<D, BWD_DVS, TA>;
    constexpr int smem_gm = (int)sizeof(BwdSmemGm<D, BWD_DVS, TA>);
    if ((e = cudaFuncSetAttribute(gk, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_gm)) != cudaSuccess)
        return e;
    gk<<<grid, 4 * BWD_DVS, smem_gm, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    auto kern = bwd_kernel<D, BWD_DVS, TA>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem1)) != cudaSuccess)
        return e;
    kern<<<dim3(a.d.hv, a.n_seqs, BWD_SEG * NS), 4 * BWD_DVS, smem1, s>>>(a);   // BWD_SEG segments per sequence
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    int blocks = (int)(a.T < (long long)sm_count() * 8 ? a.T : (long long)sm_count() * 8);
    if (blocks > 0) bwd_group_sum_kernel<<<blocks, 256, 0, s>>>(a, NS);
    return cudaGetLastError();
}

template <typename TA>
cudaError_t launch_bwd_a(const BwdArgs &a, bool states_only, cudaStream_t s) {
    switch (a.d.dk) {
        case 32: return launch_bwd_t<32, TA>(a, states_only, s);
        case 64: return launch_bwd_t<64, TA>(a, states_only, s);
        case 128: return launch_bwd_t<128, TA>(a, states_only, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

size_t bwd_ws_bytes(const Dims &d, long long T, long long n_seqs, bool states_only) {
    auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const size_t t = (size_t)(T > 0 ? T : 0), ns = (size_t)(n_seqs > 0 ? n_seqs : 0);
    const size_t nsl = (size_t)(d.dv / BWD_DVS > 0 ? d.dv / BWD_DVS : 1);
    size_t b = al((ns + 1) * 4);
    if (!states_only)
        b += al((size_t)BWD_SEG * ns * d.hv * (size_t)((d.chunk + 1) / 2) * d.dk * d.dv * 4) +
             al((size_t)(BWD_SEG - 1) * ns * d.hv * (size_t)d.dk * d.dv * 4) +
             2 * al(t * d.hv * nsl * d.dk * 4) + 3 * al(t * d.hv * nsl * 4);
    return b;
}

void bwd_carve(BwdArgs &a, void *ws, bool states_only) {
    auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
    char *p = (char *)ws;
    const size_t t = (size_t)a.T, ns = (size_t)a.n_seqs;
    const size_t nsl = (size_t)(a.d.dv / BWD_DVS > 0 ? a.d.dv / BWD_DVS : 1);
    a.chunk_base = (int *)p; p += al((ns + 1) * 4);
    if (states_only) return;
    a.scratch = (float *)p; p += al((size_t)BWD_SEG * ns * a.d.hv * (size_t)((a.d.chunk + 1) / 2) * a.d.dk * a.d.dv * 4);
    a.gsplit = (float *)p; p += al((size_t)(BWD_SEG - 1) * ns * a.d.hv * (size_t)a.d.dk * a.d.dv * 4);
    a.pq = (float *)p; p += al(t * a.d.hv * nsl * a.d.dk * 4);
    a.pk = (float *)p; p += al(t * a.d.hv * nsl * a.d.dk * 4);
    a.pda = (float *)p; p += al(t * a.d.hv * nsl * 4);
    a.pda2 = (float *)p; p += al(t * a.d.hv * nsl * 4);
    a.pdb = (float *)p;
}

cudaError_t launch_backward(const BwdArgs &a, bool in_bf16, bool states_only, cudaStream_t s) {
    if (a.n_seqs == 0) return cudaSuccess;
    return in_bf16 ? launch_bwd_a<__nv_bfloat16>(a, states_only, s)
                   : launch_bwd_a<float>(a, states_only, s);
}

}  // namespace gdn
