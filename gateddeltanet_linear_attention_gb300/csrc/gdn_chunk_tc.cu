// gdn_chunk_tc.cu -- chunked gated delta rule on the 5th-generation tensor
// cores (tcgen05, accumulators in TMEM), for dk = dv = 128 and 64-token chunks.
//
// Chunk algebra (as in the fp32 SIMT kernel; M = S^T is dk x dv, G the
// in-chunk cumulative log-decay, gamma = exp(G), chunks restart at every
// sequence start since they are relative to each invocation -- hyperflare
// core-design, GDN numerics paragraph):
//   A  = strict_lower(diag(beta) (K K^T o Gamma)),  T = (I + A)^-1
//   W  = T diag(beta gamma) K,  U = T diag(beta) V
//   U' = U - W M
//   O  = diag(gamma) Q M + (Q K^T o Gamma) U'
//   M <- gamma_last M + (diag(exp(G_last - G)) K)^T U'
//
// Precision.  The gated RMSNorm that follows divides every token-head by the
// RMS of its own o, so on quiet tokens absolute errors in o are amplified up
// to 1/sqrt(eps) = 1000x.  Single-pass bf16 operands (2^-9) fail a 1e-2
// max|dy|/RMS gate by far; every operand here is therefore split into
// bf16 hi + lo and each product is issued as hi*hi + hi*lo + lo*hi (about
// 2^-16 relative), with fp32 accumulation in TMEM and the state kept in fp32
// registers.
//
// Work decomposition: one CTA (256 threads) per (sequence, v-head, slice of
// DVS state columns); the columns of M evolve independently, so slices only
// duplicate the dv-independent products.  Per chunk, five MMA groups, all
// M = 128 (64-row problems are stacked or padded):
//   G1  D1 = [K ; Q] (128 x 128) . K^T            -> K K^T (lanes 0-63), Q K^T (64-127)
//   G2  D2 = [T ; P] (128 x 64)  . [bgK | bV]^T   -> W (cols 0-127), U (cols 128..) on lanes 0-63
//   G3  D3 = [W ; gQ] (128x128)  . M              -> W M (lanes 0-63), gamma Q M (64-127)
//   G4  D3 += [T ; P] (128 x 64) . U'             -> lanes 64-127 become O
//   G5  D5 = K~^T (128 x 64) . U'                 -> the state increment
// The triangular inverse T is formed on the SIMT pipes (four 16x16 diagonal
// blocks by forward substitution in registers, then block rows).
#include "gdn_common.cuh"
#include "tc_sm103.cuh"

namespace gdn {

namespace {

constexpr int TC_NT = 256;
constexpr int TC_C = 64;     // chunk
constexpr int TC_DK = 128;   // dk == dv

// Shared-memory map (bytes).  Every tile has a hi and a lo part.
template <int DVS>
struct TcSmem {
    static constexpr int A1 = 128 * 128 * 2;               // [K;Q] -> [W;gQ], K = 128
    static constexpr int B2 = (128 + DVS) * 64 * 2;        // [bgK | bV]^T -> K~^T (rows 0-127), K = 64
    static constexpr int A3 = 128 * 64 * 2;                // [T ; P], K = 64
    static constexpr int B3 = DVS * 128 * 2;               // M^T, K = 128
    static constexpr int B4 = DVS * 64 * 2;                // U'^T, K = 64
    static constexpr int OFF_A1 = 0;                        // hi at +0, lo at +A1
    static constexpr int OFF_B2 = OFF_A1 + 2 * A1;
    static constexpr int OFF_A3 = OFF_B2 + 2 * B2;
    static constexpr int OFF_B3 = OFF_A3 + 2 * A3;
    static constexpr int OFF_B4 = OFF_B3 + 2 * B3;
    static constexpr int OFF_SA = OFF_B4 + 2 * B4;          // fp32 A [64][65] for the solve
    static constexpr int OFF_X = OFF_SA + 64 * 65 * 4;      // fp32 scratch 3 x 16 x 17
    static constexpr int OFF_G = OFF_X + 3 * 16 * 17 * 4;   // G[64], beta[64]
    static constexpr int OFF_BAR = OFF_G + 2 * 64 * 4;      // mbarrier, tmem base, timeout flag
    static constexpr int BYTES = OFF_BAR + 16;
};

__device__ __forceinline__ void split_bf16(float v, __nv_bfloat16 &hi, __nv_bfloat16 &lo) {
    hi = __float2bfloat16_rn(v);
    lo = __float2bfloat16_rn(v - __bfloat162float(hi));
}

// Store 8 consecutive-k values of row r (k0 % 8 == 0) of a K-major tile as
// one 16-byte hi store and one 16-byte lo store.
__device__ __forceinline__ void put8(unsigned char *hi_tile, unsigned char *lo_tile, int Kdim, int r,
                                     int k0, const float *v) {
    __align__(16) __nv_bfloat16 h[8], l[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) split_bf16(v[i], h[i], l[i]);
    const uint32_t off = tc::kmaj_off(r, k0, Kdim);
    *reinterpret_cast<uint4 *>(hi_tile + off) = *reinterpret_cast<const uint4 *>(h);
    *reinterpret_cast<uint4 *>(lo_tile + off) = *reinterpret_cast<const uint4 *>(l);
}

__device__ __forceinline__ void put1(unsigned char *hi_tile, unsigned char *lo_tile, int Kdim, int r,
                                     int k, float v) {
    __nv_bfloat16 h, l;
    split_bf16(v, h, l);
    const uint32_t off = tc::kmaj_off(r, k, Kdim);
    *reinterpret_cast<__nv_bfloat16 *>(hi_tile + off) = h;
    *reinterpret_cast<__nv_bfloat16 *>(lo_tile + off) = l;
}

__device__ __forceinline__ float get1(const unsigned char *hi_tile, const unsigned char *lo_tile,
                                      int Kdim, int r, int k) {
    const uint32_t off = tc::kmaj_off(r, k, Kdim);
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(hi_tile + off)) +
           __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(lo_tile + off));
}

// Issue D (+)= A . B^T over Kdim in 16-wide steps with the three split
// products.  A: 128 rows, B: N rows, both K-major hi/lo pairs.
__device__ __forceinline__ void mma3(uint32_t d_tmem, uint32_t a_hi, uint32_t a_lo, uint32_t b_hi,
                                     uint32_t b_lo, int Kdim, uint32_t idesc, bool accumulate) {
    for (int k0 = 0; k0 < Kdim; k0 += 16) {
        const uint64_t ah = tc::kmaj_desc(a_hi, Kdim, k0), al = tc::kmaj_desc(a_lo, Kdim, k0);
        const uint64_t bh = tc::kmaj_desc(b_hi, Kdim, k0), bl = tc::kmaj_desc(b_lo, Kdim, k0);
        tc::mma_bf16(d_tmem, ah, bh, idesc, (accumulate || k0 > 0) ? 1u : 0u);
        tc::mma_bf16(d_tmem, ah, bl, idesc, 1u);
        tc::mma_bf16(d_tmem, al, bh, idesc, 1u);
    }
}

}  // namespace

template <int DVS, typename TIn, typename TOut>
__global__ void __launch_bounds__(TC_NT, 1) chunk_tc_kernel(ChunkArgs a) {
    using L = TcSmem<DVS>;
    constexpr int HALF = DVS / 2;                 // state columns per thread in lane mapping
    extern __shared__ __align__(1024) unsigned char sm[];
    unsigned char *a1h = sm + L::OFF_A1, *a1l = a1h + L::A1;
    unsigned char *b2h = sm + L::OFF_B2, *b2l = b2h + L::B2;
    unsigned char *a3h = sm + L::OFF_A3, *a3l = a3h + L::A3;
    unsigned char *b3h = sm + L::OFF_B3, *b3l = b3h + L::B3;
    unsigned char *b4h = sm + L::OFF_B4, *b4l = b4h + L::B4;
    float *sA = reinterpret_cast<float *>(sm + L::OFF_SA);     // [64][65]
    float *sX = reinterpret_cast<float *>(sm + L::OFF_X);      // [3][16][17]
    float *sG = reinterpret_cast<float *>(sm + L::OFF_G);      // [64]
    float *sB = sG + 64;                                        // [64]
    uint64_t *mbar = reinterpret_cast<uint64_t *>(sm + L::OFF_BAR);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(sm + L::OFF_BAR + 8);
    volatile uint32_t *wait_flag = reinterpret_cast<uint32_t *>(sm + L::OFF_BAR + 12);

    const Dims &d = a.d;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int slice = blockIdx.x, h = blockIdx.y, n = blockIdx.z;
    const int kh = h / d.grp;
    const int col0 = h * TC_DK + slice * DVS;      // this slice's first column in o / v / state
    // row mapping (staging): row r, column quarter cq
    const int rr = tid >> 2, cq = tid & 3;
    // lane mapping (TMEM epilogues): TMEM lane quarter qd, column half hf
    const int qd = warp & 3, hf = warp >> 2;
    const int tl = qd * 32 + lane;                 // this thread's TMEM lane / tile row

    long long s, e;
    seq_bounds(a.cu_seqlens, n, a.T, a.err, s, e);
    if (n == a.n_seqs - 1 && tid == 0 && slice == 0 && h == 0 && a.cu_seqlens[a.n_seqs] != a.T)
        set_error(a.err, GDN_DEVERR_CU_SEQLENS);
    const int slot = slot_of(a.state_idx, n, d.n_slots, a.err);
    TOut *o = (TOut *)a.o;
    const long long ldo = (long long)d.hv * TC_DK;
    if (a.state_idx && slot < 0) {
        for (long long t = s + tid / DVS; t < e; t += TC_NT / DVS)
            o[t * ldo + col0 + tid % DVS] = from_f32<TOut>(0.f);
        return;
    }

    // ---- TMEM (512 columns) and the MMA-completion barrier
    if (warp == 0) {
        tc::tmem_alloc(tc::smem_u32(tmem_slot), 512);
        tc::tmem_relinquish();
    }
    if (tid == 32) {
        tc::mbar_init(tc::smem_u32(mbar), 1);
        tc::mbar_fence_init();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tbase = *tmem_slot;
    const uint32_t T_D1 = tbase + 0, T_D2 = tbase + 64, T_D3 = tbase + 320, T_D5 = tbase + 384;
    const uint32_t lane_off = (uint32_t)(qd * 32) << 16;
    uint32_t phase = 0;
    bool timed_out = false;
    // One thread polls the MMA barrier (bounded); the block then agrees on the
    // outcome, so a timeout leaves the chunk loop uniformly.
    auto wait_mma = [&]() -> bool {
        if (tid == 0) *wait_flag = tc::mbar_wait(tc::smem_u32(mbar), phase) ? 0u : 1u;
        __syncthreads();
        const bool ok = *wait_flag == 0u;
        if (ok) phase ^= 1u;
        tc::fence_after_sync();
        return ok;
    };

    constexpr uint32_t ID_G1 = tc::idesc_bf16(128, 64);
    constexpr uint32_t ID_G2 = tc::idesc_bf16(128, 128 + DVS);
    constexpr uint32_t ID_S = tc::idesc_bf16(128, DVS);
    const uint32_t sa1h = tc::smem_u32(a1h), sa1l = tc::smem_u32(a1l);
    const uint32_t sb2h = tc::smem_u32(b2h), sb2l = tc::smem_u32(b2l);
    const uint32_t sa3h = tc::smem_u32(a3h), sa3l = tc::smem_u32(a3l);
    const uint32_t sb3h = tc::smem_u32(b3h), sb3l = tc::smem_u32(b3l);
    const uint32_t sb4h = tc::smem_u32(b4h), sb4l = tc::smem_u32(b4l);

    // ---- initial state: thread (lane tl = dk row, half hf) holds M[tl][hf*HALF ..]
    float Mr[HALF];
    {
        const float *sin = (a.state_in && slot >= 0)
                               ? a.state_in + ((long long)slot * d.hv + h) * TC_DK * TC_DK +
                                     (long long)tl * TC_DK + slice * DVS + hf * HALF
                               : nullptr;
#pragma unroll
        for (int j = 0; j < HALF; ++j) Mr[j] = sin ? sin[j] : 0.f;
#pragma unroll
        for (int j = 0; j < HALF; ++j) put1(b3h, b3l, 128, hf * HALF + j, tl, Mr[j]);
    }

    const TIn *qg = (const TIn *)a.q + (long long)kh * TC_DK;
    const TIn *kg = (const TIn *)a.k + (long long)kh * TC_DK;
    const TIn *vg = (const TIn *)a.v + col0;
    const bool l2 = (a.flags & GDN_FLAG_L2NORM_QK) != 0;
    constexpr int VQ = DVS / 4;   // v columns per thread in row mapping

    for (long long c0 = s; c0 < e; c0 += TC_C) {
        const int Lc = (int)((e - c0) < TC_C ? (e - c0) : TC_C);
        // ---------------- S0: stage row rr (32 columns of q and k, VQ of v), gates
        float kv[32], qv[32], vv[VQ];
        const bool live = rr < Lc;
        {
            const long long t = c0 + rr;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                kv[i] = live ? to_f32(kg[t * a.ld_qk + cq * 32 + i]) : 0.f;
                qv[i] = live ? to_f32(qg[t * a.ld_qk + cq * 32 + i]) : 0.f;
            }
#pragma unroll
            for (int i = 0; i < VQ; ++i) vv[i] = live ? to_f32(vg[t * a.ld_v + cq * VQ + i]) : 0.f;
        }
        if (tid < TC_C) {
            const bool lv = tid < Lc;
            sG[tid] = lv ? a.g[(c0 + tid) * d.hv + h] : 0.f;
            sB[tid] = lv ? a.beta[(c0 + tid) * d.hv + h] : 0.f;
        }
        if (l2) {
            float sk = 0.f, sq = 0.f;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                sk += kv[i] * kv[i];
                sq += qv[i] * qv[i];
            }
            sk += __shfl_xor_sync(0xffffffffu, sk, 1);
            sk += __shfl_xor_sync(0xffffffffu, sk, 2);
            sq += __shfl_xor_sync(0xffffffffu, sq, 1);
            sq += __shfl_xor_sync(0xffffffffu, sq, 2);
            const float fk = rsqrtf(sk + d.l2_eps), fq = rsqrtf(sq + d.l2_eps) * d.q_scale;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                kv[i] *= fk;
                qv[i] *= fq;
            }
        }
        __syncthreads();
        if (warp == 0) {  // inclusive scan of g over 64 rows (2 per lane); padded rows add 0
            float g0 = sG[2 * lane], g1 = sG[2 * lane + 1];
            float pair = g0 + g1, inc = pair;
#pragma unroll
            for (int o2 = 1; o2 < 32; o2 <<= 1) {
                float t2 = __shfl_up_sync(0xffffffffu, inc, o2);
                if (lane >= o2) inc += t2;
            }
            const float excl = inc - pair;
            sG[2 * lane] = excl + g0;
            sG[2 * lane + 1] = inc;
        }
        __syncthreads();
        const float Gr = sG[rr], br = sB[rr], Gl = sG[TC_C - 1];
        const float gam_r = expf(Gr), bg = br * gam_r, kdec = expf(Gl - Gr);
        // ---------------- S2: operands of G1 and G2
#pragma unroll
        for (int k8 = 0; k8 < 32; k8 += 8) {
            put8(a1h, a1l, 128, rr, cq * 32 + k8, &kv[k8]);         // K rows 0-63
            put8(a1h, a1l, 128, 64 + rr, cq * 32 + k8, &qv[k8]);    // Q rows 64-127
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) put1(b2h, b2l, 64, cq * 32 + i, rr, bg * kv[i]);   // (b g K)^T
#pragma unroll
        for (int i = 0; i < VQ; ++i) put1(b2h, b2l, 64, 128 + cq * VQ + i, rr, br * vv[i]);  // (b V)^T
        tc::fence_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        // ---------------- G1: [K;Q] K^T
        if (tid == 0) {
            mma3(T_D1, sa1h, sa1l, sa1h, sa1l, 128, ID_G1, false);
            tc::mma_commit(tc::smem_u32(mbar));
        }
        if (!wait_mma()) { timed_out = true; break; }
        // ---------------- E1: A (fp32, for the solve) and P (operand); gamma Q into A1
        {
            float v32[32];
            tc::tmem_ld32(T_D1 + lane_off + hf * 32, v32);
            const int r = tl & 63;
            const float Gq = sG[r], bq = sB[r];
            if (qd < 2) {  // K K^T rows
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int c = hf * 32 + i;
                    sA[r * 65 + c] = (c < r) ? bq * expf(Gq - sG[c]) * v32[i] : 0.f;
                }
            } else {       // Q K^T rows -> P
                float pv[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int c = hf * 32 + i;
                    pv[i] = (c <= r) ? expf(Gq - sG[c]) * v32[i] : 0.f;
                }
#pragma unroll
                for (int k8 = 0; k8 < 32; k8 += 8) put8(a3h, a3l, 64, 64 + r, hf * 32 + k8, &pv[k8]);
            }
        }
        tc::fence_before_sync();
        __syncthreads();   // G1 has finished reading A1; A is complete
        {
            float gq[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) gq[i] = gam_r * qv[i];
#pragma unroll
            for (int k8 = 0; k8 < 32; k8 += 8) put8(a1h, a1l, 128, 64 + rr, cq * 32 + k8, &gq[k8]);
        }
        // ---------------- solve T = (I + A)^-1, written as bf16 hi/lo into A3 rows 0-63
        if (warp < 4 && lane < 16) {   // diagonal 16x16 blocks, column `lane` of block `warp`
            const int b0 = warp * 16, c = lane;
            float col[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                float acc = 0.f;
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    if (i < r) acc += sA[(b0 + r) * 65 + b0 + i] * col[i];
                col[r] = (r == c) ? 1.f : ((r > c) ? -acc : 0.f);
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) put1(a3h, a3l, 64, b0 + r, b0 + c, col[r]);
        }
        __syncthreads();
        for (int bi = 1; bi < 4; ++bi) {
            // X_j = sum_{k=j}^{bi-1} A_{bi,k} T_{k,j}   for j < bi (one 16x16 block each)
            for (int idx = tid; idx < bi * 256; idx += TC_NT) {
                const int bj = idx >> 8, r = (idx >> 4) & 15, c = idx & 15;
                float acc = 0.f;
                for (int bk = bj; bk < bi; ++bk)
                    for (int m = 0; m < 16; ++m)
                        acc += sA[(bi * 16 + r) * 65 + bk * 16 + m] *
                               get1(a3h, a3l, 64, bk * 16 + m, bj * 16 + c);
                sX[(bj * 16 + r) * 17 + c] = acc;
            }
            __syncthreads();
            // T_{bi,j} = - T_{bi,bi} X_j
            for (int idx = tid; idx < bi * 256; idx += TC_NT) {
                const int bj = idx >> 8, r = (idx >> 4) & 15, c = idx & 15;
                float acc = 0.f;
                for (int m = 0; m <= r; ++m)
                    acc += get1(a3h, a3l, 64, bi * 16 + r, bi * 16 + m) * sX[(bj * 16 + m) * 17 + c];
                put1(a3h, a3l, 64, bi * 16 + r, bj * 16 + c, -acc);
            }
            __syncthreads();
        }
        // zero the strictly upper part of T's off-diagonal blocks (rows 0-63, k > row block)
        for (int idx = tid; idx < 64 * 64; idx += TC_NT) {
            const int r = idx >> 6, c = idx & 63;
            if ((c >> 4) > (r >> 4)) put1(a3h, a3l, 64, r, c, 0.f);
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        // ---------------- G2: [T;P] . [bgK | bV]^T  ->  W | U  (rows 0-63)
        if (tid == 0) {
            mma3(T_D2, sa3h, sa3l, sb2h, sb2l, 64, ID_G2, false);
            tc::mma_commit(tc::smem_u32(mbar));
        }
        if (!wait_mma()) { timed_out = true; break; }
        // ---------------- E2: W -> A1 rows 0-63, U -> registers; K~^T -> B2 rows 0-127
        float Ur[HALF];
        if (qd < 2) {
            const int r = tl;
            float v32[32];
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                tc::tmem_ld32(T_D2 + lane_off + hf * 64 + part * 32, v32);
#pragma unroll
                for (int k8 = 0; k8 < 32; k8 += 8)
                    put8(a1h, a1l, 128, r, hf * 64 + part * 32 + k8, &v32[k8]);
            }
            if (HALF == 32) {
                tc::tmem_ld32(T_D2 + lane_off + 128 + hf * HALF, v32);
#pragma unroll
                for (int j = 0; j < HALF; ++j) Ur[j] = v32[j];
            } else {
                float v16[16];
                tc::tmem_ld16(T_D2 + lane_off + 128 + hf * HALF, v16);
#pragma unroll
                for (int j = 0; j < HALF; ++j) Ur[j] = v16[j];
            }
        }
        tc::fence_before_sync();
        __syncthreads();   // G2 done with B2: overwrite rows 0-127 with K~^T
#pragma unroll
        for (int i = 0; i < 32; ++i) put1(b2h, b2l, 64, cq * 32 + i, rr, kdec * kv[i]);
        tc::fence_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        // ---------------- G3: [W ; gQ] . M
        if (tid == 0) {
            mma3(T_D3, sa1h, sa1l, sb3h, sb3l, 128, ID_S, false);
            tc::mma_commit(tc::smem_u32(mbar));
        }
        if (!wait_mma()) { timed_out = true; break; }
        // ---------------- E3: U' = U - W M  -> U'^T (B4)
        if (qd < 2) {
            float wm[HALF];
            if (HALF == 32) {
                float v32[32];
                tc::tmem_ld32(T_D3 + lane_off + hf * HALF, v32);
#pragma unroll
                for (int j = 0; j < HALF; ++j) wm[j] = v32[j];
            } else {
                float v16[16];
                tc::tmem_ld16(T_D3 + lane_off + hf * HALF, v16);
#pragma unroll
                for (int j = 0; j < HALF; ++j) wm[j] = v16[j];
            }
#pragma unroll
            for (int j = 0; j < HALF; ++j) put1(b4h, b4l, 64, hf * HALF + j, tl, Ur[j] - wm[j]);
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
        // ---------------- G4 (O += P U') and G5 (dM = K~^T U')
        if (tid == 0) {
            mma3(T_D3, sa3h, sa3l, sb4h, sb4l, 64, ID_S, true);
            mma3(T_D5, sb2h, sb2l, sb4h, sb4l, 64, ID_S, false);
            tc::mma_commit(tc::smem_u32(mbar));
        }
        if (!wait_mma()) { timed_out = true; break; }
        // ---------------- E4: outputs (lanes 64-127) and the state (all lanes)
        {
            float v[HALF];
            if (qd >= 2) {
                const int r = tl - 64;
                if (HALF == 32) {
                    float v32[32];
                    tc::tmem_ld32(T_D3 + lane_off + hf * HALF, v32);
#pragma unroll
                    for (int j = 0; j < HALF; ++j) v[j] = v32[j];
                } else {
                    float v16[16];
                    tc::tmem_ld16(T_D3 + lane_off + hf * HALF, v16);
#pragma unroll
                    for (int j = 0; j < HALF; ++j) v[j] = v16[j];
                }
                if (r < Lc) {
                    TOut *orow = o + (c0 + r) * ldo + col0 + hf * HALF;
#pragma unroll
                    for (int j = 0; j < HALF; ++j) orow[j] = from_f32<TOut>(v[j]);
                }
            }
            if (HALF == 32) {
                float v32[32];
                tc::tmem_ld32(T_D5 + lane_off + hf * HALF, v32);
#pragma unroll
                for (int j = 0; j < HALF; ++j) v[j] = v32[j];
            } else {
                float v16[16];
                tc::tmem_ld16(T_D5 + lane_off + hf * HALF, v16);
#pragma unroll
                for (int j = 0; j < HALF; ++j) v[j] = v16[j];
            }
            const float gl = expf(Gl);
#pragma unroll
            for (int j = 0; j < HALF; ++j) {
                Mr[j] = gl * Mr[j] + v[j];
                put1(b3h, b3l, 128, hf * HALF + j, tl, Mr[j]);
            }
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
    }
    if (timed_out) {
        // give the outstanding MMAs one more bounded chance to retire before TMEM is freed
        if (tid == 0) {
            set_error(a.err, GDN_DEVERR_TIMEOUT);
            tc::mbar_wait(tc::smem_u32(mbar), phase);
        }
        __syncthreads();
    }
    if (a.state_out && slot >= 0) {
        float *so = a.state_out + ((long long)slot * d.hv + h) * TC_DK * TC_DK +
                    (long long)tl * TC_DK + slice * DVS + hf * HALF;
#pragma unroll
        for (int j = 0; j < HALF; ++j) so[j] = Mr[j];
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tbase, 512);
}

template <int DVS, typename TIn, typename TOut>
static cudaError_t launch_tc_t(const ChunkArgs &a, cudaStream_t s) {
    auto kern = chunk_tc_kernel<DVS, TIn, TOut>;
    constexpr int smem = TcSmem<DVS>::BYTES;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    dim3 grid(TC_DK / DVS, a.d.hv, a.n_seqs);
    kern<<<grid, TC_NT, smem, s>>>(a);
    return cudaGetLastError();
}

bool chunk_tc_supported(const Dims &d) { return d.dk == 128 && d.dv == 128 && d.chunk == 64; }

cudaError_t launch_chunk_tc(const ChunkArgs &a, bool in_bf16, bool o_bf16, int dvs, cudaStream_t s) {
    if (a.n_seqs == 0) return cudaSuccess;
    if (!chunk_tc_supported(a.d)) return cudaErrorInvalidValue;
#define GDN_TC(DVS_)                                                                         \
    if (dvs == DVS_) {                                                                        \
        if (in_bf16)                                                                          \
            return o_bf16 ? launch_tc_t<DVS_, __nv_bfloat16, __nv_bfloat16>(a, s)             \
                          : launch_tc_t<DVS_, __nv_bfloat16, float>(a, s);                    \
        return o_bf16 ? launch_tc_t<DVS_, float, __nv_bfloat16>(a, s)                         \
                      : launch_tc_t<DVS_, float, float>(a, s);                                \
    }
    GDN_TC(32)
    GDN_TC(64)
#undef GDN_TC
    return cudaErrorInvalidValue;
}

}  // namespace gdn
