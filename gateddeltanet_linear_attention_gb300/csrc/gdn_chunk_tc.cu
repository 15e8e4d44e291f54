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
//   G1  D1 = [K ; Q] . K^T               -> K K^T (TMEM lanes 0-63), Q K^T (64-127)
//   G2  D2 = [T ; P] . [bgK | bV]        -> W (cols 0-127) | U on lanes 0-63
//   G3  D3 = [W ; gQ] . M                -> W M (lanes 0-63), gamma Q M (64-127)
//   G4  D3 += [T ; P] . U'               -> lanes 64-127 become O
//   G5  D5 = K~^T . U'                   -> the state increment
// Operands whose contraction index is the token or the dk row (bgK|bV, K~,
// M, U') are stored MN-major, so that every operand is written from its
// natural row layout with 16-byte stores.  The triangular inverse T is formed
// in fp32 on the SIMT pipes (four 16x16 diagonal blocks by forward
// substitution in registers, then block rows), with T kept transposed in the
// unused upper triangle of A.
#include "gdn_common.cuh"
#include "tc_sm103.cuh"

namespace gdn {

namespace {

constexpr int TC_NT = 256;
constexpr int TC_C = 64;     // chunk
constexpr int TC_DK = 128;   // dk == dv

// Shared-memory map (bytes).  Every bf16 tile has a hi part and a lo part.
template <int DVS>
struct TcSmem {
    static constexpr int NB = 128 + DVS;                   // N of G2's B operand
    static constexpr int KQ = 128 * 128 * 2;               // [K;Q] -> [W;gQ], K-major, K = 128
    static constexpr int BW = NB * 64 * 2;                 // [bgK|bV] MN-major (MN = NB, K = 64) -> K~ (MN = 128)
    static constexpr int TP = 128 * 64 * 2;                // [T ; P], K-major, K = 64
    static constexpr int MT = DVS * 128 * 2;               // M, MN-major (MN = DVS, K = 128)
    static constexpr int UT = DVS * 64 * 2;                // U', MN-major (MN = DVS, K = 64)
    static constexpr int OFF_KQ = 0;
    static constexpr int OFF_BW = OFF_KQ + 2 * KQ;
    static constexpr int OFF_TP = OFF_BW + 2 * BW;
    static constexpr int OFF_MT = OFF_TP + 2 * TP;
    static constexpr int OFF_UT = OFF_MT + 2 * MT;
    static constexpr int OFF_SA = OFF_UT + 2 * UT;          // fp32 [64][65]: A below, T^T above the diagonal
    static constexpr int OFF_GAM = OFF_SA + 64 * 65 * 4;    // fp32 [64][65]: exp(G_r - G_c), c <= r
    static constexpr int OFF_X = OFF_GAM + 64 * 65 * 4;     // (reserved)
    static constexpr int OFF_G = OFF_X + 16;                // G[64], beta[64]
    static constexpr int OFF_BAR = OFF_G + 2 * 64 * 4;      // mbarrier, tmem base, timeout flag
    static constexpr int BYTES = OFF_BAR + 16;
};

// Store 8 values at byte offset `off` (16-byte aligned) of a hi and a lo tile
// (packed two-at-a-time conversions).
__device__ __forceinline__ void put8(unsigned char *hi, unsigned char *lo, uint32_t off, const float *v) {
    __nv_bfloat162 h2[4], l2[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        h2[i] = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
        const float2 hf = __bfloat1622float2(h2[i]);
        l2[i] = __floats2bfloat162_rn(v[2 * i] - hf.x, v[2 * i + 1] - hf.y);
    }
    *reinterpret_cast<uint4 *>(hi + off) = *reinterpret_cast<const uint4 *>(h2);
    *reinterpret_cast<uint4 *>(lo + off) = *reinterpret_cast<const uint4 *>(l2);
}

// Read back 8 values (hi + lo) at a 16-byte aligned offset of a hi and a lo tile.
__device__ __forceinline__ void get8(const unsigned char *hi, const unsigned char *lo, uint32_t off, float *v) {
    const uint4 hv = *reinterpret_cast<const uint4 *>(hi + off);
    const uint4 lv = *reinterpret_cast<const uint4 *>(lo + off);
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&hv);
    const __nv_bfloat162 *l = reinterpret_cast<const __nv_bfloat162 *>(&lv);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 a = __bfloat1622float2(h[i]), b = __bfloat1622float2(l[i]);
        v[2 * i] = a.x + b.x;
        v[2 * i + 1] = a.y + b.y;
    }
}

// Load n (multiple of 8) consecutive elements as fp32 with 16-byte loads.
template <int n>
__device__ __forceinline__ void load_row(const float *p, float *out) {
#pragma unroll
    for (int i = 0; i < n; i += 4) {
        const float4 v = *reinterpret_cast<const float4 *>(p + i);
        out[i] = v.x; out[i + 1] = v.y; out[i + 2] = v.z; out[i + 3] = v.w;
    }
}
template <int n>
__device__ __forceinline__ void load_row(const __nv_bfloat16 *p, float *out) {
#pragma unroll
    for (int i = 0; i < n; i += 8) {
        const uint4 v = *reinterpret_cast<const uint4 *>(p + i);
        const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(&v);
#pragma unroll
        for (int j = 0; j < 8; ++j) out[i + j] = __bfloat162float(b[j]);
    }
}

template <int n>
__device__ __forceinline__ void store_row(float *p, const float *v) {
#pragma unroll
    for (int i = 0; i < n; i += 4) *reinterpret_cast<float4 *>(p + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
}
template <int n>
__device__ __forceinline__ void store_row(__nv_bfloat16 *p, const float *v) {
#pragma unroll
    for (int i = 0; i < n; i += 8) {
        __align__(16) __nv_bfloat16 b[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) b[j] = __float2bfloat16_rn(v[i + j]);
        *reinterpret_cast<uint4 *>(p + i) = *reinterpret_cast<const uint4 *>(b);
    }
}

template <int n>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, float *v) {
    if constexpr (n == 32) {
        float t[32];
        tc::tmem_ld32(taddr, t);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = t[i];
    } else {
        static_assert(n == 16, "16 or 32 columns");
        float t[16];
        tc::tmem_ld16(taddr, t);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = t[i];
    }
}

// Issue D (+)= A . B over Kdim in 16-wide steps with the three split
// products.  A_MN / B_MN select MN-major operands (with their MN extent).
template <bool A_MN, bool B_MN>
__device__ __forceinline__ void mma3(uint32_t d_tmem, uint32_t a_hi, uint32_t a_lo, uint32_t a_mn,
                                     uint32_t b_hi, uint32_t b_lo, uint32_t b_mn, int Kdim,
                                     uint32_t idesc, bool accumulate) {
    for (int k0 = 0; k0 < Kdim; k0 += 16) {
        const uint64_t ah = A_MN ? tc::mnmaj_desc(a_hi, a_mn, k0) : tc::kmaj_desc(a_hi, Kdim, k0);
        const uint64_t al = A_MN ? tc::mnmaj_desc(a_lo, a_mn, k0) : tc::kmaj_desc(a_lo, Kdim, k0);
        const uint64_t bh = B_MN ? tc::mnmaj_desc(b_hi, b_mn, k0) : tc::kmaj_desc(b_hi, Kdim, k0);
        const uint64_t bl = B_MN ? tc::mnmaj_desc(b_lo, b_mn, k0) : tc::kmaj_desc(b_lo, Kdim, k0);
        tc::mma_bf16(d_tmem, ah, bh, idesc, (accumulate || k0 > 0) ? 1u : 0u);
        tc::mma_bf16(d_tmem, ah, bl, idesc, 1u);
        tc::mma_bf16(d_tmem, al, bh, idesc, 1u);
    }
}

// One block of the triangular inverse, for the block column held by a warp:
// rows of block bi = bj + DB, column m of T, from the rows already in tcol.
// (Lanes c and c+16 hold the same column; each stores half of the new rows.)
template <int DB>
__device__ __forceinline__ void solve_block_col(float *sA, float (&tcol)[48], int bj, int m, int rh) {
    // Blocks past the last row block are computed on clamped (valid) addresses
    // and not stored, so that the warp's code has no data-dependent branches.
    const bool live = bj + DB < 4;
    const int bi = live ? bj + DB : 3;
    float xr[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        const float *arow = sA + (bi * 16 + r) * 65 + bj * 16;
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < 16 * DB; ++k) acc = fmaf(arow[k], tcol[k], acc);
        xr[r] = acc;
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) {
        float acc = xr[r];
#pragma unroll
        for (int mm = 0; mm < r; ++mm) acc = fmaf(sA[(bi * 16 + mm) * 65 + bi * 16 + r], xr[mm], acc);
        tcol[16 * DB + r] = -acc;
    }
    if (live) {
#pragma unroll
        for (int r = 0; r < 8; ++r) sA[m * 65 + bi * 16 + rh * 8 + r] = tcol[16 * DB + rh * 8 + r];
    }
}

}  // namespace

template <int DVS, typename TIn, typename TOut>
__global__ void __launch_bounds__(TC_NT, 1) chunk_tc_kernel(ChunkArgs a) {
    using L = TcSmem<DVS>;
    constexpr int HALF = DVS / 2;                 // state columns per thread in lane mapping
    constexpr int VQ = DVS / 4;                   // v columns per thread in row mapping
    constexpr int NB = L::NB;
    extern __shared__ __align__(1024) unsigned char sm[];
    unsigned char *kqh = sm + L::OFF_KQ, *kql = kqh + L::KQ;
    unsigned char *bwh = sm + L::OFF_BW, *bwl = bwh + L::BW;
    unsigned char *tph = sm + L::OFF_TP, *tpl = tph + L::TP;
    unsigned char *mth = sm + L::OFF_MT, *mtl = mth + L::MT;
    unsigned char *uth = sm + L::OFF_UT, *utl = uth + L::UT;
    float *sA = reinterpret_cast<float *>(sm + L::OFF_SA);     // [64][65]
    float *sGam = reinterpret_cast<float *>(sm + L::OFF_GAM);  // [64][65]
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
    // row mapping (staging): row rr, column quarter cq
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
    auto sync_for_mma = [&]() {   // generic smem writes -> visible to the tensor core
        tc::fence_async_smem();
        tc::fence_before_sync();
        __syncthreads();
        tc::fence_after_sync();
    };

    constexpr uint32_t ID_G1 = tc::idesc_bf16(128, 64);
    constexpr uint32_t ID_G2 = tc::idesc_bf16(128, NB) | tc::kTransB;
    constexpr uint32_t ID_G34 = tc::idesc_bf16(128, DVS) | tc::kTransB;
    constexpr uint32_t ID_G5 = tc::idesc_bf16(128, DVS) | tc::kTransA | tc::kTransB;
    const uint32_t s_kqh = tc::smem_u32(kqh), s_kql = tc::smem_u32(kql);
    const uint32_t s_bwh = tc::smem_u32(bwh), s_bwl = tc::smem_u32(bwl);
    const uint32_t s_tph = tc::smem_u32(tph), s_tpl = tc::smem_u32(tpl);
    const uint32_t s_mth = tc::smem_u32(mth), s_mtl = tc::smem_u32(mtl);
    const uint32_t s_uth = tc::smem_u32(uth), s_utl = tc::smem_u32(utl);

    // ---- initial state: thread (lane tl = dk row, half hf) holds M[tl][hf*HALF ..]
    float Mr[HALF];
    {
        if (a.state_in && slot >= 0) {
            const float *sin = a.state_in + ((long long)slot * d.hv + h) * TC_DK * TC_DK +
                               (long long)tl * TC_DK + slice * DVS + hf * HALF;
            load_row<HALF>(sin, Mr);
        } else {
#pragma unroll
            for (int j = 0; j < HALF; ++j) Mr[j] = 0.f;
        }
#pragma unroll
        for (int j8 = 0; j8 < HALF; j8 += 8) put8(mth, mtl, tc::mnmaj_off(hf * HALF + j8, tl, DVS), &Mr[j8]);
    }

    const TIn *qg = (const TIn *)a.q + (long long)kh * TC_DK + cq * 32;
    const TIn *kg = (const TIn *)a.k + (long long)kh * TC_DK + cq * 32;
    const TIn *vg = (const TIn *)a.v + col0 + cq * VQ;
    const bool l2 = (a.flags & GDN_FLAG_L2NORM_QK) != 0;

    // Raw rows of the chunk at c0 (row rr of the row mapping) and its gates: the
    // loads of chunk c+1 are issued while chunk c's second MMA group runs.
    float kv[32], qv[32], vv[VQ];
    auto load_chunk = [&](long long c0) {
        const long long t = c0 + rr;
        if (t < e) {
            load_row<32>(kg + t * a.ld_qk, kv);
            load_row<32>(qg + t * a.ld_qk, qv);
            load_row<VQ>(vg + t * a.ld_v, vv);
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) kv[i] = qv[i] = 0.f;
#pragma unroll
            for (int i = 0; i < VQ; ++i) vv[i] = 0.f;
        }
    };
    float gn = 0.f, bn = 0.f;     // gates of the next chunk (threads tid < 64)
    auto load_gates = [&](long long c0) {
        if (tid < TC_C) {
            const long long t = c0 + tid;
            gn = t < e ? a.g[t * d.hv + h] : 0.f;
            bn = t < e ? a.beta[t * d.hv + h] : 0.f;
        }
    };
    if (s < e) {
        load_chunk(s);
        load_gates(s);
        if (tid < TC_C) {
            sG[tid] = gn;
            sB[tid] = bn;
        }
    }

    for (long long c0 = s; c0 < e; c0 += TC_C) {
        const int Lc = (int)((e - c0) < TC_C ? (e - c0) : TC_C);
        const bool has_next = c0 + TC_C < e;
        // ---------------- S0: L2 norm of the staged rows; gate scan
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
        __syncthreads();   // raw gates of this chunk are in sG / sB
        if (warp == 0) {   // inclusive scan of g over 64 rows (2 per lane); padded rows add 0
            const float g0 = sG[2 * lane], g1 = sG[2 * lane + 1];
            const float pair = g0 + g1;
            float inc = pair;
#pragma unroll
            for (int o2 = 1; o2 < 32; o2 <<= 1) {
                const float t2 = __shfl_up_sync(0xffffffffu, inc, o2);
                if (lane >= o2) inc += t2;
            }
            sG[2 * lane] = inc - pair + g0;
            sG[2 * lane + 1] = inc;
        }
        __syncthreads();
        const float Gr = sG[rr], br = sB[rr], Gl = sG[TC_C - 1];
        const float bg = br * expf(Gr);
        // ---------------- S2: operands of G1 (K and Q rows) and G2 ([bgK | bV], MN-major)
#pragma unroll
        for (int k8 = 0; k8 < 32; k8 += 8) {
            put8(kqh, kql, tc::kmaj_off(rr, cq * 32 + k8, 128), &kv[k8]);
            put8(kqh, kql, tc::kmaj_off(64 + rr, cq * 32 + k8, 128), &qv[k8]);
            float t8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) t8[i] = bg * kv[k8 + i];
            put8(bwh, bwl, tc::mnmaj_off(cq * 32 + k8, rr, NB), t8);
        }
#pragma unroll
        for (int k8 = 0; k8 < VQ; k8 += 8) {
            float t8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) t8[i] = br * vv[k8 + i];
            put8(bwh, bwl, tc::mnmaj_off(128 + cq * VQ + k8, rr, NB), t8);
        }
        sync_for_mma();
        // ---------------- G1: [K;Q] K^T;  meanwhile the decay table
        if (tid == 0) {
            mma3<false, false>(T_D1, s_kqh, s_kql, 0, s_kqh, s_kql, 0, 128, ID_G1, false);
            tc::mma_commit(tc::smem_u32(mbar));
        }
        {
            const float Gq = sG[rr];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int c = cq * 16 + i;
                sGam[rr * 65 + c] = (c <= rr) ? expf(Gq - sG[c]) : 0.f;
            }
        }
        if (!wait_mma()) { timed_out = true; break; }
        // ---------------- E1: A (fp32, for the solve), P (operand), gamma Q in place
        {
            float v32[32];
            tc::tmem_ld32(T_D1 + lane_off + hf * 32, v32);
            const int r = tl & 63;
            const float *grow = sGam + r * 65 + hf * 32;
            if (qd < 2) {  // K K^T rows -> A (strictly lower)
                const float bq = sB[r];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int c = hf * 32 + i;
                    if (c < r) sA[r * 65 + c] = bq * grow[i] * v32[i];
                }
            } else {       // Q K^T rows -> P (lower incl. diagonal; Gamma is 0 above)
#pragma unroll
                for (int i = 0; i < 32; ++i) v32[i] *= grow[i];
#pragma unroll
                for (int k8 = 0; k8 < 32; k8 += 8) put8(tph, tpl, tc::kmaj_off(64 + r, hf * 32 + k8, 64), &v32[k8]);
            }
        }
        {   // G1 is done with Q: replace it by gamma Q (read back hi + lo)
            const float gam_r = expf(Gr);
#pragma unroll
            for (int k8 = 0; k8 < 32; k8 += 8) {
                float t8[8];
                const uint32_t off = tc::kmaj_off(64 + rr, cq * 32 + k8, 128);
                get8(kqh, kql, off, t8);
#pragma unroll
                for (int i = 0; i < 8; ++i) t8[i] *= gam_r;
                put8(kqh, kql, off, t8);
            }
        }
        __syncthreads();
        // ---------------- solve T = (I + A)^-1: diagonal 16x16 blocks (column `lane` of block `warp`)
        if (warp < 4 && lane < 16) {
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
            for (int r = 0; r < 16; ++r)
                if (r > c) sA[(b0 + c) * 65 + b0 + r] = col[r];   // T[b0+r][b0+c], stored transposed
        }
        __syncthreads();
        // Off-diagonal blocks, one warp per block column bj (no barriers inside):
        // T[bi][bj] = -T[bi][bi] . sum_{k=bj}^{bi-1} A[bi][k] T[k][bj]   for bi > bj.
        if (warp < 3) {
            const int bj = warp, c = lane & 15, rh = lane >> 4;
            const int m = bj * 16 + c;
            float tcol[48];   // T[16*bj + k][m], k < 48
#pragma unroll
            for (int k = 0; k < 48; ++k) {
                const int row = bj * 16 + k;
                tcol[k] = (k < 16) ? ((row > m) ? sA[m * 65 + row] : ((row == m) ? 1.f : 0.f)) : 0.f;
            }
            solve_block_col<1>(sA, tcol, bj, m, rh);
            solve_block_col<2>(sA, tcol, bj, m, rh);
            solve_block_col<3>(sA, tcol, bj, m, rh);
        }
        __syncthreads();
        // T -> bf16 hi/lo, rows 0-63 of TP (K-major): 64 rows x 8 groups of 8 columns
        for (int task = tid; task < 64 * 8; task += TC_NT) {
            const int r = task >> 3, c8 = (task & 7) * 8;
            float t8[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int c = c8 + i;
                t8[i] = (c < r) ? sA[c * 65 + r] : ((c == r) ? 1.f : 0.f);
            }
            put8(tph, tpl, tc::kmaj_off(r, c8, 64), t8);
        }
        sync_for_mma();
        // ---------------- G2: [T;P] . [bgK | bV]  ->  W | U  (rows 0-63); meanwhile the
        // next chunk's rows and gates are loaded (after the shared-memory-heavy solve, so
        // that the global loads do not queue in front of it)
        if (tid == 0) {
            mma3<false, true>(T_D2, s_tph, s_tpl, 0, s_bwh, s_bwl, NB, 64, ID_G2, false);
            tc::mma_commit(tc::smem_u32(mbar));
        }
        if (has_next) {
            load_chunk(c0 + TC_C);
            load_gates(c0 + TC_C);
        }
        if (!wait_mma()) { timed_out = true; break; }
        // ---------------- E2a: K~ = exp(G_last - G_r) K_r (MN-major A of G5) into the freed B2
        // region; K is read back (hi + lo) from KQ rows 0-63 before W replaces it
        {
            const float kdec = expf(Gl - Gr);
#pragma unroll
            for (int k8 = 0; k8 < 32; k8 += 8) {
                float t8[8];
                get8(kqh, kql, tc::kmaj_off(rr, cq * 32 + k8, 128), t8);
#pragma unroll
                for (int i = 0; i < 8; ++i) t8[i] *= kdec;
                put8(bwh, bwl, tc::mnmaj_off(cq * 32 + k8, rr, 128), t8);
            }
        }
        __syncthreads();
        // ---------------- E2b: W -> rows 0-63 of KQ (G1 is done with K), U -> registers
        float Ur[HALF];
        if (qd < 2) {
            float v32[32];
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                tc::tmem_ld32(T_D2 + lane_off + hf * 64 + part * 32, v32);
#pragma unroll
                for (int k8 = 0; k8 < 32; k8 += 8)
                    put8(kqh, kql, tc::kmaj_off(tl, hf * 64 + part * 32 + k8, 128), &v32[k8]);
            }
            tmem_ld<HALF>(T_D2 + lane_off + 128 + hf * HALF, Ur);
        }
        sync_for_mma();
        // ---------------- G3: [W ; gQ] . M
        if (tid == 0) {
            mma3<false, true>(T_D3, s_kqh, s_kql, 0, s_mth, s_mtl, DVS, 128, ID_G34, false);
            tc::mma_commit(tc::smem_u32(mbar));
        }
        if (!wait_mma()) { timed_out = true; break; }
        // ---------------- E3: U' = U - W M  -> MN-major B operand
        if (qd < 2) {
            float wm[HALF];
            tmem_ld<HALF>(T_D3 + lane_off + hf * HALF, wm);
#pragma unroll
            for (int j = 0; j < HALF; ++j) wm[j] = Ur[j] - wm[j];
#pragma unroll
            for (int j8 = 0; j8 < HALF; j8 += 8) put8(uth, utl, tc::mnmaj_off(hf * HALF + j8, tl, DVS), &wm[j8]);
        }
        sync_for_mma();
        // ---------------- G4 (O += P U') and G5 (dM = K~^T U'); meanwhile the next chunk's gates
        if (tid == 0) {
            mma3<false, true>(T_D3, s_tph, s_tpl, 0, s_uth, s_utl, DVS, 64, ID_G34, true);
            mma3<true, true>(T_D5, s_bwh, s_bwl, 128, s_uth, s_utl, DVS, 64, ID_G5, false);
            tc::mma_commit(tc::smem_u32(mbar));
        }
        if (has_next && tid < TC_C) {
            sG[tid] = gn;
            sB[tid] = bn;
        }
        if (!wait_mma()) { timed_out = true; break; }
        // ---------------- E4: outputs (lanes 64-127) and the state (all lanes)
        {
            float v[HALF];
            if (qd >= 2) {
                const int r = tl - 64;
                tmem_ld<HALF>(T_D3 + lane_off + hf * HALF, v);
                if (r < Lc) store_row<HALF>(o + (c0 + r) * ldo + col0 + hf * HALF, v);
            }
            tmem_ld<HALF>(T_D5 + lane_off + hf * HALF, v);
            const float gl = expf(Gl);
#pragma unroll
            for (int j = 0; j < HALF; ++j) Mr[j] = gl * Mr[j] + v[j];
#pragma unroll
            for (int j8 = 0; j8 < HALF; j8 += 8) put8(mth, mtl, tc::mnmaj_off(hf * HALF + j8, tl, DVS), &Mr[j8]);
        }
        // (the next chunk's first operand writes are followed by sync_for_mma before G1)
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
        store_row<HALF>(so, Mr);
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
#undef GDN_TC
    return cudaErrorInvalidValue;
}

}  // namespace gdn
