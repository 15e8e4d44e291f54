// gdn_chunk_simt.cu -- chunked gated delta rule in fp32 on the SIMT pipes.
//
// This is the fp32-input path (and the exact-arithmetic companion of the
// tensor-core kernel).  Chunk algebra, with M = S^T (dk x dv), G_r the
// cumulative log-decay inside a chunk of Lc tokens (restarting at each
// sequence start, as chunks are relative to each invocation -- hyperflare
// core-design, GDN numerics paragraph) and gamma_r = exp(G_r):
//   A[r][i]  = beta_r exp(G_r - G_i) k_r.k_i               (i < r)
//   (I + A) U' = diag(beta) (V - diag(gamma) K M)           forward substitution
//   O        = diag(gamma) Q M + (Q K^T o Gamma) U'         Gamma[r][i] = exp(G_r - G_i), i <= r
//   M       <- gamma_last M + (diag(exp(G_last - G_r)) K)^T U'
// Decay ratios are only ever formed as exp(G_r - G_i) with i <= r, so nothing
// overflows however strong the decay.
//
// Parallelism: one CTA per (sequence, v-head, 32-column slice of dv).  The
// columns of M evolve independently given K, so slices need no exchange; the
// q.k and k.k products are recomputed per slice.  The state slice lives in
// shared memory for the whole sequence and is read from / written to HBM
// once.
#include "gdn_common.cuh"

namespace gdn {

constexpr int SIMT_DVS = 32;   // dv columns per CTA
constexpr int SIMT_NT = 256;

template <int DK, int C>
struct SimtSmem {
    static constexpr int KP = DK + 1;       // padded row pitch of K and Q
    static constexpr int AP = C + 1;        // padded row pitch of the C x C matrices
    float K[C * KP];
    float Q[C * KP];
    float U[C * SIMT_DVS];                  // V -> right-hand side -> U'
    float O[C * SIMT_DVS];                  // gamma * Q M, then the output rows
    float A[C * AP];                        // beta_r Gamma k_r.k_i  (strictly lower)
    float P[C * AP];                        // Gamma q_r.k_i         (lower incl. diagonal)
    float M[DK * SIMT_DVS];
    float G[C], beta[C];
};

template <typename T>
__device__ __forceinline__ const T *cptr(const void *p) { return (const T *)p; }

template <int DK, int C, typename TIn, typename TOut>
__global__ void __launch_bounds__(SIMT_NT) chunk_simt_kernel(ChunkArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    using SM = SimtSmem<DK, C>;
    SM &sm = *reinterpret_cast<SM *>(smem_raw);
    constexpr int KP = SM::KP, AP = SM::AP, DVS = SIMT_DVS;
    const Dims &d = a.d;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int slice = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int kh = h / d.grp;
    const int col0 = h * d.dv + slice * DVS;  // column of this slice in o / v

    long long s, e;
    seq_bounds(a.cu_seqlens, n, a.T, a.err, s, e);
    if (n == a.n_seqs - 1 && tid == 0 && slice == 0 && h == 0 && a.cu_seqlens[a.n_seqs] != a.T)
        set_error(a.err, GDN_DEVERR_CU_SEQLENS);
    int slot = slot_of(a.state_idx, n, d.n_slots, a.err);
    TOut *o = (TOut *)a.o;
    if (a.state_idx && slot < 0) {  // padding lane: zero outputs, no state traffic
        for (long long t = s; t < e; ++t)
            for (int j = tid; j < DVS; j += SIMT_NT) o[t * d.hv * d.dv + col0 + j] = from_f32<TOut>(0.f);
        return;
    }
    // initial state slice
    const float *sin = (a.state_in && slot >= 0)
                           ? a.state_in + ((long long)slot * d.hv + h) * DK * d.dv + slice * DVS
                           : nullptr;
    for (int idx = tid; idx < DK * DVS; idx += SIMT_NT) {
        int i = idx / DVS, j = idx % DVS;
        sm.M[idx] = sin ? sin[(long long)i * d.dv + j] : 0.f;
    }

    const TIn *qg = cptr<TIn>(a.q) + (long long)kh * DK;
    const TIn *kg = cptr<TIn>(a.k) + (long long)kh * DK;
    const TIn *vg = cptr<TIn>(a.v) + col0;
    const bool l2 = (a.flags & GDN_FLAG_L2NORM_QK) != 0;

    for (long long c0 = s; c0 < e; c0 += C) {
        const int Lc = (int)((e - c0) < C ? (e - c0) : C);
        __syncthreads();  // previous chunk fully consumed
        // ---- stage the chunk: K, Q rows (head kh), V slice, gates
        for (int idx = tid; idx < C * DK; idx += SIMT_NT) {
            int r = idx / DK, i = idx % DK;
            float kv = 0.f, qv = 0.f;
            if (r < Lc) {
                kv = to_f32(kg[(c0 + r) * a.ld_qk + i]);
                qv = to_f32(qg[(c0 + r) * a.ld_qk + i]);
            }
            sm.K[r * KP + i] = kv;
            sm.Q[r * KP + i] = qv;
        }
        for (int idx = tid; idx < C * DVS; idx += SIMT_NT) {
            int r = idx / DVS, j = idx % DVS;
            sm.U[idx] = r < Lc ? to_f32(vg[(c0 + r) * a.ld_v + j]) : 0.f;
        }
        if (tid < C) {
            float gv = 0.f, bv = 0.f;
            if (tid < Lc) {
                gv = a.g[(c0 + tid) * d.hv + h];
                bv = a.beta[(c0 + tid) * d.hv + h];
            }
            sm.G[tid] = gv;
            sm.beta[tid] = bv;
        }
        __syncthreads();
        if (tid == 0) {  // inclusive cumulative log-decay; padded rows repeat the last value
            float acc = 0.f;
            for (int r = 0; r < C; ++r) {
                acc += sm.G[r];
                sm.G[r] = acc;
            }
        }
        if (l2) {  // per-row L2 norm of q and k (q also scaled)
            for (int r = warp; r < 2 * C; r += SIMT_NT / 32) {
                float *row = (r < C) ? &sm.K[r * KP] : &sm.Q[(r - C) * KP];
                float ss = 0.f;
                for (int i = lane; i < DK; i += 32) ss += row[i] * row[i];
                ss = warp_sum(ss);
                float sc = rsqrtf(ss + d.l2_eps);
                if (r >= C) sc *= d.q_scale;
                for (int i = lane; i < DK; i += 32) row[i] *= sc;
            }
        }
        __syncthreads();
        // ---- A and P (TB x TB register tiles over a 16 x 16 thread grid), K M and Q M
        {
            constexpr int TB = C / 16;
            const int r0 = (tid / 16) * TB, i0 = (tid % 16) * TB;
            float kk[TB][TB] = {}, qk[TB][TB] = {};
            for (int e2 = 0; e2 < DK; ++e2) {
                float kr[TB], qr[TB], ki[TB];
#pragma unroll
                for (int x = 0; x < TB; ++x) {
                    kr[x] = sm.K[(r0 + x) * KP + e2];
                    qr[x] = sm.Q[(r0 + x) * KP + e2];
                    ki[x] = sm.K[(i0 + x) * KP + e2];
                }
#pragma unroll
                for (int x = 0; x < TB; ++x)
#pragma unroll
                    for (int y = 0; y < TB; ++y) {
                        kk[x][y] += kr[x] * ki[y];
                        qk[x][y] += qr[x] * ki[y];
                    }
            }
#pragma unroll
            for (int x = 0; x < TB; ++x)
#pragma unroll
                for (int y = 0; y < TB; ++y) {
                    int r = r0 + x, i = i0 + y;
                    float dec = (i <= r) ? expf(sm.G[r] - sm.G[i]) : 0.f;
                    sm.A[r * AP + i] = (i < r) ? sm.beta[r] * dec * kk[x][y] : 0.f;
                    sm.P[r * AP + i] = (i <= r) ? dec * qk[x][y] : 0.f;
                }
        }
        {
            const int j = lane, rb = warp * (C / 8);
            constexpr int RPW = C / 8;
            float km[RPW], qm[RPW];
#pragma unroll
            for (int x = 0; x < RPW; ++x) km[x] = qm[x] = 0.f;
            for (int i = 0; i < DK; ++i) {
                float m = sm.M[i * DVS + j];
#pragma unroll
                for (int x = 0; x < RPW; ++x) {
                    km[x] += sm.K[(rb + x) * KP + i] * m;
                    qm[x] += sm.Q[(rb + x) * KP + i] * m;
                }
            }
#pragma unroll
            for (int x = 0; x < RPW; ++x) {
                int r = rb + x;
                float gam = expf(sm.G[r]);
                sm.U[r * DVS + j] = sm.beta[r] * (sm.U[r * DVS + j] - gam * km[x]);
                sm.O[r * DVS + j] = gam * qm[x];
            }
        }
        __syncthreads();
        // ---- forward substitution (I + A) U' = rhs, 8 lanes per column
        {
            const int j = warp * 4 + (lane >> 3), sub = lane & 7;
            for (int r = 1; r < Lc; ++r) {
                float part = 0.f;
                for (int i = sub; i < r; i += 8) part += sm.A[r * AP + i] * sm.U[i * DVS + j];
                part += __shfl_xor_sync(0xffffffffu, part, 4);
                part += __shfl_xor_sync(0xffffffffu, part, 2);
                part += __shfl_xor_sync(0xffffffffu, part, 1);
                if (sub == 0) sm.U[r * DVS + j] -= part;
                __syncwarp();
            }
        }
        __syncthreads();
        // ---- outputs O += P U'
        {
            const int j = lane, rb = warp * (C / 8);
            for (int x = 0; x < C / 8; ++x) {
                int r = rb + x;
                if (r >= Lc) break;
                float acc = sm.O[r * DVS + j];
                for (int i = 0; i <= r; ++i) acc += sm.P[r * AP + i] * sm.U[i * DVS + j];
                o[(c0 + r) * d.hv * d.dv + col0 + j] = from_f32<TOut>(acc);
            }
        }
        // ---- state M <- gamma_last M + (diag(exp(G_last - G_r)) K)^T U'
        {
            const int j = lane;
            constexpr int RPT = DK / 8;
            const int ib = warp * RPT;
            const float gl = sm.G[Lc - 1];
            float m[RPT];
            const float gam = expf(gl);
#pragma unroll
            for (int x = 0; x < RPT; ++x) m[x] = gam * sm.M[(ib + x) * DVS + j];
            for (int r = 0; r < Lc; ++r) {
                float u = sm.U[r * DVS + j] * expf(gl - sm.G[r]);
#pragma unroll
                for (int x = 0; x < RPT; ++x) m[x] += sm.K[r * KP + ib + x] * u;
            }
#pragma unroll
            for (int x = 0; x < RPT; ++x) sm.M[(ib + x) * DVS + j] = m[x];
        }
    }
    __syncthreads();
    if (a.state_out && slot >= 0) {
        float *so = a.state_out + ((long long)slot * d.hv + h) * DK * d.dv + slice * DVS;
        for (int idx = tid; idx < DK * DVS; idx += SIMT_NT) {
            int i = idx / DVS, j = idx % DVS;
            so[(long long)i * d.dv + j] = sm.M[idx];
        }
    }
}

template <int DK, int C, typename TIn, typename TOut>
static cudaError_t launch_simt_t(const ChunkArgs &a, cudaStream_t s) {
    auto kern = chunk_simt_kernel<DK, C, TIn, TOut>;
    size_t smem = sizeof(SimtSmem<DK, C>);
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem);
    if (err != cudaSuccess) return err;
    dim3 grid(a.d.dv / SIMT_DVS, a.d.hv, a.n_seqs);
    kern<<<grid, SIMT_NT, smem, s>>>(a);
    return cudaGetLastError();
}

template <int DK, int C>
static cudaError_t launch_simt_dt(const ChunkArgs &a, bool in_bf16, bool o_bf16, cudaStream_t s) {
    if (in_bf16) {
        return o_bf16 ? launch_simt_t<DK, C, __nv_bfloat16, __nv_bfloat16>(a, s)
                      : launch_simt_t<DK, C, __nv_bfloat16, float>(a, s);
    }
    return o_bf16 ? launch_simt_t<DK, C, float, __nv_bfloat16>(a, s)
                  : launch_simt_t<DK, C, float, float>(a, s);
}

cudaError_t launch_chunk_simt(const ChunkArgs &a, bool in_bf16, bool o_bf16, cudaStream_t s) {
    if (a.n_seqs == 0) return cudaSuccess;
    const int dk = a.d.dk, C = a.d.chunk;
#define GDN_SIMT(DK_, C_) \
    if (dk == DK_ && C == C_) return launch_simt_dt<DK_, C_>(a, in_bf16, o_bf16, s)
    GDN_SIMT(32, 16);
    GDN_SIMT(32, 64);
    GDN_SIMT(64, 16);
    GDN_SIMT(64, 64);
    GDN_SIMT(128, 16);
    GDN_SIMT(128, 64);
#undef GDN_SIMT
    return cudaErrorInvalidValue;
}

}  // namespace gdn
