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
// Two launches and a reduction:
//  - bwd_states_kernel (gdn_chunk_states): one CTA per (sequence, v-head,
//    slice), the forward over the sequence with the slice of M in registers
//    (thread: one float4 column group over RPT rows, 8 lanes per 128-byte row
//    segment), writing it at every chunk start: the states a training forward
//    retains;
//  - bwd_kernel (gdn_chunk_backward): one CTA per (sequence, v-head, slice),
//    the chunks in reverse: the forward of the chunk from its boundary state,
//    keeping the state before every token in the workspace, then the tokens in
//    reverse with GM in registers.  Column sums go through one shared-memory
//    pass, row sums through shuffles among the lanes that hold the row;
//  - bwd_group_sum_kernel adds the slices and the v-heads of each q/k head
//    (dq, dk) and the slices of each v-head (dg = a (<GM, M> - beta dw . p),
//    dbeta).
#include "gdn_common.cuh"

namespace gdn {

namespace {

// DV here is the slice width (32 columns); a thread holds 4 columns of RPT rows.
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

// Per-token inputs of one v-head staged in shared memory.
// One token's inputs in shared memory (double-buffered: the next token's are stored while this
// one's are read).  Every array read or written as float4 is 16-byte aligned explicitly.
template <int DK, int DV>
struct TokIn {
    alignas(16) float q[DK];
    alignas(16) float k[DK];
    alignas(16) float v[DV];
    alignas(16) float dout[DV];
    float a, b;
};
template <int DK, int DV>
struct TokSmem {
    TokIn<DK, DV> in[2];
    alignas(16) float p[DV];
    alignas(16) float r[DV];
    alignas(16) float w[DV];
    alignas(16) float dp[DV];
    alignas(16) float red[BwdCfg<DK, DV>::RPP][DV];
    float wsum[3][BwdCfg<DK, DV>::NT / 32];
};

// A thread's share of one token's inputs, loaded into registers ahead of use: k and q for
// tid < DK, v and do for tid < DV, a and beta for thread 0.
struct TokReg {
    float k, q, v, dout, a, b;
};

// The forward step of one token on M in registers: p = M^T k (column sums), w, M <- a M + k w^T.
// `after_first_barrier` runs once every thread is past the first barrier (the other input
// buffer is free then).
template <int DK, int DV, typename F>
__device__ __forceinline__ void fwd_token(float4 (&m)[BwdCfg<DK, DV>::RPT], TokSmem<DK, DV> &sm,
                                          const TokIn<DK, DV> &in, int tid, int rg, int c4,
                                          F after_first_barrier) {
    using C = BwdCfg<DK, DV>;
    float4 pp = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int x = 0; x < C::RPT; ++x) {
        const float kr = in.k[rg + x * C::RPP];
        pp.x += m[x].x * kr; pp.y += m[x].y * kr; pp.z += m[x].z * kr; pp.w += m[x].w * kr;
    }
    *reinterpret_cast<float4 *>(&sm.red[rg][c4]) = pp;
    __syncthreads();
    after_first_barrier();
    if (tid < DV) {
        float p = 0.f;
#pragma unroll
        for (int r = 0; r < C::RPP; ++r) p += sm.red[r][tid];
        sm.w[tid] = in.b * (in.v[tid] - in.a * p);
    }
    __syncthreads();
    const float4 w4 = *reinterpret_cast<const float4 *>(&sm.w[c4]);
    const float a = in.a;
#pragma unroll
    for (int x = 0; x < C::RPT; ++x) {
        const float kr = in.k[rg + x * C::RPP];
        m[x].x = a * m[x].x + kr * w4.x; m[x].y = a * m[x].y + kr * w4.y;
        m[x].z = a * m[x].z + kr * w4.z; m[x].w = a * m[x].w + kr * w4.w;
    }
}

// Token t's q (optional), k, v, do (optional), a, beta of head h: the thread's share into
// registers, and from there into an input buffer.
template <int DK, int DV, typename TA>
__device__ __forceinline__ TokReg load_token(const BwdArgs &a, long long t, int h, int kh, int tid,
                                             bool with_q, int col0) {
    TokReg r = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (tid < DK) {
        r.k = to_f32(((const TA *)a.k)[t * a.ld_qk + (long long)kh * DK + tid]);
        if (with_q) r.q = to_f32(((const TA *)a.q)[t * a.ld_qk + (long long)kh * DK + tid]);
    }
    if (tid < DV) {   // the slice's columns col0 .. col0 + DV of the head
        r.v = to_f32(((const TA *)a.v)[t * a.ld_v + (long long)h * a.d.dv + col0 + tid]);
        if (with_q) r.dout = a.d_o[t * (long long)a.d.hv * a.d.dv + (long long)h * a.d.dv + col0 + tid];
    }
    if (tid == 0) {
        r.a = a.g[t * a.d.hv + h];
        r.b = a.beta[t * a.d.hv + h];
    }
    return r;
}
template <int DK, int DV>
__device__ __forceinline__ void store_token(TokIn<DK, DV> &in, const TokReg &r, int tid) {
    static_assert(DK <= BwdCfg<DK, DV>::NT, "one k / q element per thread");
    if (tid < DK) { in.k[tid] = r.k; in.q[tid] = r.q; }
    if (tid < DV) { in.v[tid] = r.v; in.dout[tid] = r.dout; }
    if (tid == 0) { in.a = expf(r.a); in.b = r.b; }
}

template <int DK, int DV, typename TA>
__global__ void __launch_bounds__(4 * DV) bwd_states_kernel(BwdArgs a) {
    using C = BwdCfg<DK, DV>;
    __shared__ __align__(16) TokSmem<DK, DV> sm;
    const Dims &d = a.d;
    const int tid = threadIdx.x, h = blockIdx.x, n = blockIdx.y, kh = h / d.grp;
    const int col0 = blockIdx.z * DV;                   // this CTA's slice of the state columns
    const int rg = tid / C::LPR, c4 = (tid % C::LPR) * 4 + col0;   // (c4: column in the head)
    const int c4s = c4 - col0;                          //         (column in the slice)
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
    store_token<DK, DV>(sm.in[0], load_token<DK, DV, TA>(a, s, h, kh, tid, false, col0), tid);
    __syncthreads();
    for (long long t = s; t < e; ++t) {
        if ((t - s) % Cc == 0) {
            float *B = a.bnd + ((b0 + (t - s) / Cc) * d.hv + h) * DK * DVH;
#pragma unroll
            for (int x = 0; x < C::RPT; ++x)
                *reinterpret_cast<float4 *>(B + (long long)(rg + x * C::RPP) * DVH + c4) = m[x];
        }
        // token t+1's inputs load while token t runs; they go to the other buffer once it is free
        const bool more = t + 1 < e;
        TokReg nx = {};
        if (more) nx = load_token<DK, DV, TA>(a, t + 1, h, kh, tid, false, col0);
        const int bi = (int)((t - s) & 1);
        fwd_token<DK, DV>(m, sm, sm.in[bi], tid, rg, c4s, [&] {
            if (more) store_token<DK, DV>(sm.in[bi ^ 1], nx, tid);
        });
    }
}

template <int DK, int DV, typename TA>
__global__ void __launch_bounds__(4 * DV) bwd_kernel(BwdArgs a) {
    using C = BwdCfg<DK, DV>;
    constexpr int NW = C::NT / 32;
    __shared__ __align__(16) TokSmem<DK, DV> sm;
    const Dims &d = a.d;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int h = blockIdx.x, n = blockIdx.y, kh = h / d.grp;
    const int sl = blockIdx.z, NS = gridDim.z, col0 = sl * DV;   // this CTA's slice of the columns
    const int rg = tid / C::LPR, c4s = (tid % C::LPR) * 4, c4 = c4s + col0;
    long long s, e;
    seq_bounds(a.cu_seqlens, n, a.T, a.err, s, e);
    const int slot = slot_of(a.state_idx, n, d.n_slots, a.err);
    const int DVH = d.dv;
    const long long HVDV = (long long)d.hv * DVH;
    auto part = [&](long long t) { return (t * d.hv + h) * NS + sl; };   // index of this slice's parts
    if (slot < 0) {                                      // padding lane: zero gradients
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
    float4 gm[C::RPT];
#pragma unroll
    for (int x = 0; x < C::RPT; ++x) {
        gm[x] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (a.d_state_out)
            gm[x] = *reinterpret_cast<const float4 *>(a.d_state_out + ((long long)slot * d.hv + h) * DK * DVH +
                                                      (long long)(rg + x * C::RPP) * DVH + c4);
    }
    // this CTA's scratch: the slice of the state before each token of one chunk
    float *scr = a.scratch + (((long long)n * d.hv + h) * NS + sl) * (long long)Cc * DK * DV;
    const long long b0 = a.chunk_base[n];
    const long long nch = (e - s + Cc - 1) / Cc;
    for (long long c = nch - 1; c >= 0; --c) {
        const long long t0 = s + c * Cc, t1 = (t0 + Cc < e) ? t0 + Cc : e;
        float4 m[C::RPT];
        {
            const float *B = a.bnd + ((b0 + c) * d.hv + h) * DK * DVH;
#pragma unroll
            for (int x = 0; x < C::RPT; ++x)
                m[x] = *reinterpret_cast<const float4 *>(B + (long long)(rg + x * C::RPP) * DVH + c4);
        }
        // forward through the chunk, keeping the state before every token (each thread
        // reads back only what it wrote); token inputs double-buffered (buffer (t - t0) & 1)
        __syncthreads();                                 // the previous chunk's buffer reads are done
        if (t0 + 1 < t1) store_token<DK, DV>(sm.in[0], load_token<DK, DV, TA>(a, t0, h, kh, tid, false, col0), tid);
        __syncthreads();
        for (long long t = t0; t < t1; ++t) {
            float *Sc = scr + (t - t0) * DK * DV;
#pragma unroll
            for (int x = 0; x < C::RPT; ++x)
                *reinterpret_cast<float4 *>(Sc + (long long)(rg + x * C::RPP) * DV + c4s) = m[x];
            if (t + 1 == t1) break;
            const bool more = t + 2 < t1;               // token t+1 updates the state too
            TokReg nx = {};
            if (more) nx = load_token<DK, DV, TA>(a, t + 1, h, kh, tid, false, col0);
            const int bi = (int)((t - t0) & 1);
            fwd_token<DK, DV>(m, sm, sm.in[bi], tid, rg, c4s, [&] {
                if (more) store_token<DK, DV>(sm.in[bi ^ 1], nx, tid);
            });
        }
        // the tokens in reverse, inputs double-buffered (buffer (t - t0) & 1): token t-1's load
        // while token t runs and are stored to the other buffer after barrier (A)
        __syncthreads();                                 // the forward pass's buffer reads are done
        store_token<DK, DV>(sm.in[(t1 - 1 - t0) & 1], load_token<DK, DV, TA>(a, t1 - 1, h, kh, tid, true, col0), tid);
        __syncthreads();
        for (long long t = t1 - 1; t >= t0; --t) {
            const float *Sc = scr + (t - t0) * DK * DV;
#pragma unroll
            for (int x = 0; x < C::RPT; ++x)
                m[x] = *reinterpret_cast<const float4 *>(Sc + (long long)(rg + x * C::RPP) * DV + c4s);
            const int bi = (int)((t - t0) & 1);
            const TokIn<DK, DV> &in = sm.in[bi];
            const bool more = t - 1 >= t0;
            TokReg nx = {};
            if (more) nx = load_token<DK, DV, TA>(a, t - 1, h, kh, tid, true, col0);
            // p = M^T k
            {
                float4 pp = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int x = 0; x < C::RPT; ++x) {
                    const float kr = in.k[rg + x * C::RPP];
                    pp.x += m[x].x * kr; pp.y += m[x].y * kr; pp.z += m[x].z * kr; pp.w += m[x].w * kr;
                }
                *reinterpret_cast<float4 *>(&sm.red[rg][c4s]) = pp;
            }
            __syncthreads();                             // (A) the other buffer is free from here
            if (more) store_token<DK, DV>(sm.in[bi ^ 1], nx, tid);
            const float av = in.a, bv = in.b;
            if (tid < DV) {
                float p = 0.f;
#pragma unroll
                for (int r = 0; r < C::RPP; ++r) p += sm.red[r][tid];
                const float rr = in.v[tid] - av * p;
                sm.p[tid] = p;
                sm.r[tid] = rr;
                sm.w[tid] = bv * rr;
            }
            __syncthreads();                             // (B)
            const float4 w4 = *reinterpret_cast<const float4 *>(&sm.w[c4s]);
            const float4 do4 = *reinterpret_cast<const float4 *>(&in.dout[c4s]);
            float4 dwp = make_float4(0.f, 0.f, 0.f, 0.f);
            float dap = 0.f;
#pragma unroll
            for (int x = 0; x < C::RPT; ++x) {
                const int row = rg + x * C::RPP;
                const float kr = in.k[row], qr = in.q[row];
                float4 mp;                               // M' = a M + k w^T
                mp.x = av * m[x].x + kr * w4.x; mp.y = av * m[x].y + kr * w4.y;
                mp.z = av * m[x].z + kr * w4.z; mp.w = av * m[x].w + kr * w4.w;
                gm[x].x += qr * do4.x; gm[x].y += qr * do4.y; gm[x].z += qr * do4.z; gm[x].w += qr * do4.w;
                const float dq = row_sum<C::LPR>(mp.x * do4.x + mp.y * do4.y + mp.z * do4.z + mp.w * do4.w);
                if (lane % C::LPR == 0) a.pq[part(t) * DK + row] = dq;
                dwp.x += gm[x].x * kr; dwp.y += gm[x].y * kr; dwp.z += gm[x].z * kr; dwp.w += gm[x].w * kr;
                dap += gm[x].x * m[x].x + gm[x].y * m[x].y + gm[x].z * m[x].z + gm[x].w * m[x].w;
            }
            *reinterpret_cast<float4 *>(&sm.red[rg][c4s]) = dwp;
            dap = warp_sum(dap);
            if (lane == 0) sm.wsum[0][warp] = dap;
            __syncthreads();                             // (C)
            if (tid < DV) {
                float dw = 0.f;
#pragma unroll
                for (int r = 0; r < C::RPP; ++r) dw += sm.red[r][tid];
                a.dv[t * HVDV + (long long)h * DVH + col0 + tid] = bv * dw;
                sm.dp[tid] = -av * bv * dw;
                const float db = warp_sum(dw * sm.r[tid]);
                const float da2 = warp_sum(dw * sm.p[tid]);
                if (lane == 0) { sm.wsum[1][warp] = db; sm.wsum[2][warp] = da2; }
            }
            __syncthreads();                             // (D)
            if (tid == 0) {   // this slice's parts of <GM, M>, dw . p and dw . r
                float da = 0.f, db = 0.f, da2 = 0.f;
                for (int wi = 0; wi < NW; ++wi) da += sm.wsum[0][wi];
                for (int wi = 0; wi < DV / 32; ++wi) { db += sm.wsum[1][wi]; da2 += sm.wsum[2][wi]; }
                a.pda[part(t)] = da;
                a.pda2[part(t)] = da2;
                a.pdb[part(t)] = db;
            }
            const float4 dp4 = *reinterpret_cast<const float4 *>(&sm.dp[c4s]);
#pragma unroll
            for (int x = 0; x < C::RPT; ++x) {
                const int row = rg + x * C::RPP;
                const float kr = in.k[row];
                const float dk = row_sum<C::LPR>(gm[x].x * w4.x + gm[x].y * w4.y + gm[x].z * w4.z +
                                                 gm[x].w * w4.w + m[x].x * dp4.x + m[x].y * dp4.y +
                                                 m[x].z * dp4.z + m[x].w * dp4.w);
                if (lane % C::LPR == 0) a.pk[part(t) * DK + row] = dk;
                gm[x].x = av * gm[x].x + kr * dp4.x; gm[x].y = av * gm[x].y + kr * dp4.y;
                gm[x].z = av * gm[x].z + kr * dp4.z; gm[x].w = av * gm[x].w + kr * dp4.w;
            }
        }
    }
    if (a.d_state_in) {
        float *D = a.d_state_in + ((long long)slot * d.hv + h) * DK * DVH;
#pragma unroll
        for (int x = 0; x < C::RPT; ++x)
            *reinterpret_cast<float4 *>(D + (long long)(rg + x * C::RPP) * DVH + c4) = gm[x];
    }
}

// dq, dk of each q/k head: the sum over its v-heads and their column slices; dg and dbeta of
// each v-head from its slices' parts (dg = a (<GM, M> - beta dw . p)).
__global__ void bwd_group_sum_kernel(BwdArgs a, int NS) {
    const Dims &d = a.d;
    const long long total = a.T * d.hk * d.dk;
    for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
         e += (long long)gridDim.x * blockDim.x) {
        const long long t = e / (d.hk * d.dk);
        const int rem = (int)(e - t * d.hk * d.dk), kh = rem / d.dk, i = rem % d.dk;
        float sq = 0.f, sk = 0.f;
        for (int gi = 0; gi < d.grp; ++gi)
            for (int sl = 0; sl < NS; ++sl) {
                const long long src = ((t * d.hv + kh * d.grp + gi) * NS + sl) * d.dk + i;
                sq += a.pq[src];
                sk += a.pk[src];
            }
        a.dq[t * a.ld_dqk + (long long)kh * d.dk + i] = sq;
        a.dk[t * a.ld_dqk + (long long)kh * d.dk + i] = sk;
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
    if (states_only) {
        bwd_states_kernel<D, BWD_DVS, TA><<<grid, 4 * BWD_DVS, 0, s>>>(a);
        return cudaGetLastError();
    }
    bwd_kernel<D, BWD_DVS, TA><<<grid, 4 * BWD_DVS, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    long long total = a.T * a.d.hk * a.d.dk;
    int blocks = (int)((total + 255) / 256);
    if (blocks > sm_count() * 16) blocks = sm_count() * 16;
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
        b += al(ns * d.hv * (size_t)d.chunk * d.dk * d.dv * 4) + 2 * al(t * d.hv * nsl * d.dk * 4) +
             3 * al(t * d.hv * nsl * 4);
    return b;
}

void bwd_carve(BwdArgs &a, void *ws, bool states_only) {
    auto al = [](size_t x) { return (x + 255) & ~(size_t)255; };
    char *p = (char *)ws;
    const size_t t = (size_t)a.T, ns = (size_t)a.n_seqs;
    const size_t nsl = (size_t)(a.d.dv / BWD_DVS > 0 ? a.d.dv / BWD_DVS : 1);
    a.chunk_base = (int *)p; p += al((ns + 1) * 4);
    if (states_only) return;
    a.scratch = (float *)p; p += al(ns * a.d.hv * (size_t)a.d.chunk * a.d.dk * a.d.dv * 4);
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
