// gdn_decode.cu -- one-token recurrent update of the gated delta rule.
//
// Per sequence n and v-head h, with M = S^T (dk x dv, fp32) and one token:
//   p = M^T k,  s = M^T q                    (one pass over M)
//   u' = beta (v - a p)
//   o  = a s + u' (k.q)                       (= M_new^T q)
//   M <- a M + k u'^T                         (written once)
// which is S <- a S (I - b k k^T) + b v k^T, o = S q, rearranged so that the
// state is read once and written once (haskell-infer-demo README,
// kernels/fla_gdn.cu "recurrent decode"; the state is the FP32 recurrence of
// hyperflare core-design's serving-defaults table).
//
// The kernel is HBM-bound: 2 * dk * dv * 4 bytes per head per token.  Layout
// of the work: one CTA per (sequence, q/k head), looping over the v-heads
// that share that q/k head.  Thread t owns 4 consecutive columns (one float4)
// of RPT rows; a warp covers whole 512-byte rows, so every state load and
// store is a fully coalesced 16-byte vector access.  Column sums over rows go
// through registers, then one shared-memory pass over the 16 row groups.
//
// decode_kernel below serves gdn_recurrent_decode (q, k, v, g, beta given);
// the fused mixer decode (conv step, gates and gated RMSNorm included) is the
// prep + streaming pair further down.
#include "gdn_common.cuh"
#include "tc_sm103.cuh"

namespace gdn {

template <int DK, int DV>
struct DecodeCfg {
    static constexpr int NT = 4 * DV;          // threads per CTA
    static constexpr int LPR = DV / 4;         // threads per state row
    static constexpr int RPP = NT / LPR;       // rows covered per pass (16)
    static constexpr int RPT = DK / RPP;       // rows per thread
    static constexpr int MAXG = 4;             // largest GQA group
};

template <int DK, int DV, typename TA, typename TOut>
__global__ void __launch_bounds__(4 * DV) decode_kernel(DecodeArgs a) {
    using Cfg = DecodeCfg<DK, DV>;
    constexpr int NT = Cfg::NT, LPR = Cfg::LPR, RPP = Cfg::RPP, RPT = Cfg::RPT;
    __shared__ __align__(16) float qs[DK];
    __shared__ __align__(16) float ks[DK];
    __shared__ __align__(16) float vs[Cfg::MAXG][DV];
    __shared__ float gate_a[Cfg::MAXG], gate_b[Cfg::MAXG];
    __shared__ __align__(16) float red_p[RPP][DV];
    __shared__ __align__(16) float red_s[RPP][DV];
    __shared__ __align__(16) float up[DV];
    __shared__ __align__(16) float os[DV];
    __shared__ float scal[8];

    const Dims &d = a.d;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = blockIdx.x / d.hk, kh = blockIdx.x % d.hk;
    const int G = d.grp;
    const int slot = slot_of(a.state_idx, n, d.n_slots, a.err);
    TOut *out = (TOut *)a.out;
    const long long out_row = (long long)n * d.hv * DV;

    if (slot < 0) {  // padding lane: zero output rows, no state or history traffic
        for (int idx = tid; idx < G * DV; idx += NT)
            out[out_row + (long long)kh * G * DV + idx] = from_f32<TOut>(0.f);
        return;
    }

    const int rg = tid / LPR;            // row group: rows rg, rg+RPP, ...
    const int c4 = (tid % LPR) * 4;      // first of this thread's 4 columns
    float *Mbase = a.state + ((long long)slot * d.hv + (long long)kh * G) * DK * DV;

    // issue the first head's state loads before the prologue
    float4 m[RPT];
#pragma unroll
    for (int x = 0; x < RPT; ++x)
        m[x] = *reinterpret_cast<const float4 *>(Mbase + (long long)(rg + x * RPP) * DV + c4);

    // ---- prologue: q, k (this q/k head) and v (its v-heads), gates
    {
        const TA *q = (const TA *)a.q + (long long)n * a.ld_qk + (long long)kh * DK;
        const TA *k = (const TA *)a.k + (long long)n * a.ld_qk + (long long)kh * DK;
        const TA *v = (const TA *)a.v + (long long)n * a.ld_v + (long long)kh * G * DV;
        for (int i = tid; i < DK; i += NT) {
            qs[i] = to_f32(q[i]);
            ks[i] = to_f32(k[i]);
        }
        for (int idx = tid; idx < G * DV; idx += NT) vs[idx / DV][idx % DV] = to_f32(v[idx]);
        if (tid < G) {
            const int h = kh * G + tid;
            gate_a[tid] = expf(a.g[(long long)n * d.hv + h]);
            gate_b[tid] = a.beta[(long long)n * d.hv + h];
        }
    }
    __syncthreads();
    const bool l2 = (a.flags & GDN_FLAG_L2NORM_QK) != 0;
    if (warp < 2) {  // warp 0: |q|, warp 1: |k|
        float *vec = warp == 0 ? qs : ks;
        float ss = 0.f;
        for (int i = lane; i < DK; i += 32) ss += vec[i] * vec[i];
        ss = warp_sum(ss);
        if (lane == 0) scal[warp] = ss;
    }
    __syncthreads();
    if (l2) {
        const float sq = rsqrtf(scal[0] + d.l2_eps) * d.q_scale, sk = rsqrtf(scal[1] + d.l2_eps);
        for (int i = tid; i < DK; i += NT) {
            qs[i] *= sq;
            ks[i] *= sk;
        }
        __syncthreads();
    }
    if (warp == 0) {  // k.q after normalisation
        float kq = 0.f;
        for (int i = lane; i < DK; i += 32) kq += ks[i] * qs[i];
        kq = warp_sum(kq);
        if (lane == 0) scal[2] = kq;
    }
    float kr[RPT], qr[RPT];
#pragma unroll
    for (int x = 0; x < RPT; ++x) {
        kr[x] = ks[rg + x * RPP];
        qr[x] = qs[rg + x * RPP];
    }

    for (int gi = 0; gi < G; ++gi) {
        const int h = kh * G + gi;
        float *Mh = Mbase + (long long)gi * DK * DV;
        if (gi > 0) {
#pragma unroll
            for (int x = 0; x < RPT; ++x)
                m[x] = *reinterpret_cast<const float4 *>(Mh + (long long)(rg + x * RPP) * DV + c4);
        }
        // column partial sums over this thread's rows
        float4 pp = make_float4(0.f, 0.f, 0.f, 0.f), ss = pp;
#pragma unroll
        for (int x = 0; x < RPT; ++x) {
            pp.x += m[x].x * kr[x]; pp.y += m[x].y * kr[x]; pp.z += m[x].z * kr[x]; pp.w += m[x].w * kr[x];
            ss.x += m[x].x * qr[x]; ss.y += m[x].y * qr[x]; ss.z += m[x].z * qr[x]; ss.w += m[x].w * qr[x];
        }
        *reinterpret_cast<float4 *>(&red_p[rg][c4]) = pp;
        *reinterpret_cast<float4 *>(&red_s[rg][c4]) = ss;
        __syncthreads();
        const float ga = gate_a[gi], gb = gate_b[gi];
        if (tid < DV) {
            float p = 0.f, s = 0.f;
#pragma unroll
            for (int r = 0; r < RPP; ++r) {
                p += red_p[r][tid];
                s += red_s[r][tid];
            }
            float u = gb * (vs[gi][tid] - ga * p);
            up[tid] = u;
            os[tid] = ga * s + u * scal[2];
        }
        __syncthreads();
        // state update, written once
        {
            const float4 u4 = *reinterpret_cast<const float4 *>(&up[c4]);
#pragma unroll
            for (int x = 0; x < RPT; ++x) {
                float4 mn;
                mn.x = ga * m[x].x + kr[x] * u4.x;
                mn.y = ga * m[x].y + kr[x] * u4.y;
                mn.z = ga * m[x].z + kr[x] * u4.z;
                mn.w = ga * m[x].w + kr[x] * u4.w;
                *reinterpret_cast<float4 *>(Mh + (long long)(rg + x * RPP) * DV + c4) = mn;
            }
        }
        // output row of this v-head
        if (tid < DV) out[out_row + (long long)h * DV + tid] = from_f32<TOut>(os[tid]);
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Fused decode, the product path: two launches.
//
// decode_prep_kernel (one CTA per (sequence, q/k head) unit, all units in
// parallel): the conv step of the unit's q/k channels and of its G v-heads'
// channels (each history has exactly one owner, so the in-place shift is
// race-free), SiLU, the q/k L2 norm, k.q, the gates and SiLU(z), written as one
// record per unit to the caller's workspace.  Doing this for every unit at
// once pays the global-load latency once, instead of on the state stream's
// critical path.
//
// decode_stream_kernel (persistent, one CTA per SM): walks its units; each
// unit's G head states (dk*dv*4 bytes each) flow HBM -> shared memory through
// a ring of NS slots filled by bulk asynchronous copies (cp.async.bulk,
// completion counted on one mbarrier per slot), so that while one head is
// updated the next NS-1 are in flight.  The records of the next batch of HB
// heads are bulk-copied into shared memory one batch ahead, so each head
// touches only shared memory before its state is written back.
// GM: the v-heads per q/k head the register arrays are sized for (1, 2 or 4; d.grp <= GM).
template <int DK, int DV, typename TA, int GM>
__global__ void __launch_bounds__(256, 8) decode_prep_kernel(DecodeArgs a) {
    __shared__ __align__(16) float qs[DK], ks[DK];
    __shared__ float scal[8 + 8];
    const Dims &d = a.d;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // The streaming kernel may be scheduled as soon as every prep CTA has
    // started: it cannot share an SM with one, and it waits for this grid's
    // completion (griddepcontrol.wait) before it reads any record.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int u = blockIdx.x, n = u / d.hk, kh = u % d.hk, G = d.grp;
    const DecRec R(DK, DV, G);
    float *rec = a.ws + (long long)u * R.size;
    const int slot = slot_of(a.state_idx, n, d.n_slots, a.err);
    if (slot < 0) {
        if (tid == 0) rec[R.slot] = __int_as_float(-1);
        return;
    }
    const TA *x = (const TA *)a.x + (long long)n * a.ld_x;
    const TA *w = (const TA *)a.conv_w;
    TA *cs = (TA *)a.conv_state + (long long)slot * d.ch * 3;
    const int nch = 2 * DK + G * DV;
    // Every global load of the unit is issued before any store (the stores to the history and
    // the record could alias later loads for the compiler, which would serialise the round trips).
    constexpr int CPT = (2 * DK + GM * DV + 255) / 256;  // channels per thread
    constexpr int ZPT = (GM * DV + 255) / 256;           // SiLU(z) values per thread
    TA hx[CPT][4], zr[ZPT];
    typename TapVec<TA>::type wv[CPT];
    int chan[CPT];
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int ci = tid + 256 * i;
        int c = 0;
        if (ci < DK) c = kh * DK + ci;
        else if (ci < 2 * DK) c = d.hk * DK + kh * DK + (ci - DK);
        else c = 2 * d.hk * DK + kh * G * DV + (ci - 2 * DK);
        chan[i] = c;
        if (ci < nch) {
            const TA *hc = cs + (long long)c * 3;
            hx[i][0] = hc[0];
            hx[i][1] = hc[1];
            hx[i][2] = hc[2];
            hx[i][3] = x[c];
            wv[i] = load_taps(w, c);
        }
    }
    const TA *z = (const TA *)a.z + (long long)n * a.ld_z + (long long)kh * G * DV;
#pragma unroll
    for (int i = 0; i < ZPT; ++i)
        if (tid + 256 * i < G * DV) zr[i] = z[tid + 256 * i];
    TA ul = from_f32<TA>(0.f), bl = from_f32<TA>(0.f);
    float alog = 0.f, dtb = 0.f;
    if (tid < G) {
        ul = ((const TA *)a.u + (long long)n * a.ld_ub)[kh * G + tid];
        bl = ((const TA *)a.b_logit + (long long)n * a.ld_ub)[kh * G + tid];
        alog = a.A_log[kh * G + tid];
        dtb = a.dt_bias[kh * G + tid];
    }
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int ci = tid + 256 * i;
        if (ci >= nch) break;
        TA *hc = cs + (long long)chan[i] * 3;
        float t[4];
        taps_f32(wv[i], t);
        const float acc = t[0] * to_f32(hx[i][0]) + t[1] * to_f32(hx[i][1]) + t[2] * to_f32(hx[i][2]) +
                          t[3] * to_f32(hx[i][3]);
        hc[0] = hx[i][1];
        hc[1] = hx[i][2];
        hc[2] = hx[i][3];
        const float val = silu_f(acc);
        if (ci < DK) qs[ci] = val;
        else if (ci < 2 * DK) ks[ci - DK] = val;
        else rec[R.v + (ci - 2 * DK)] = val;
    }
#pragma unroll
    for (int i = 0; i < ZPT; ++i)
        if (tid + 256 * i < G * DV) rec[R.z + tid + 256 * i] = silu_f(to_f32(zr[i]));
    if (tid < G) {
        const float gg = -expf(alog) * softplus_f(to_f32(ul) + dtb);
        rec[R.ga + tid] = expf(gg);
        rec[R.gb + tid] = sigmoid_f(to_f32(bl));
    }
    __syncthreads();
    if (warp < 2) {   // |q|^2 (warp 0), |k|^2 (warp 1)
        const float *vec = warp == 0 ? qs : ks;
        float ss = 0.f;
        for (int i = lane; i < DK; i += 32) ss += vec[i] * vec[i];
        ss = warp_sum(ss);
        if (lane == 0) scal[warp] = ss;
    }
    __syncthreads();
    const float fq = rsqrtf(scal[0] + d.l2_eps) * d.q_scale, fk = rsqrtf(scal[1] + d.l2_eps);
    float kq = 0.f;
    for (int i = tid; i < DK; i += 256) {
        const float qn = qs[i] * fq, kn = ks[i] * fk;
        rec[R.q + i] = qn;
        rec[R.k + i] = kn;
        kq += qn * kn;
    }
    kq = warp_sum(kq);
    if (lane == 0) scal[8 + warp] = kq;
    __syncthreads();
    if (tid == 0) {
        float t = 0.f;
        for (int wi = 0; wi < 8; ++wi) t += scal[8 + wi];
        rec[R.kq] = t;
        rec[R.slot] = __int_as_float(slot);
    }
}

// ---- Q8 state codec (used by the streaming kernel in its Q8 form and by
// q8_convert_kernel; the format is described with gdn_state_to_q8 below)
// The hash's output step from its state (state = v * 747796405 + 2891336453).
__device__ __forceinline__ uint32_t pcg_output(uint32_t state) {
    const uint32_t word = ((state >> ((state >> 28u) + 4u)) ^ state) * 277803737u;
    return (word >> 22u) ^ word;
}
__device__ __forceinline__ uint32_t pcg_hash(uint32_t v) { return pcg_output(v * 747796405u + 2891336453u); }

template <int L>
__device__ __forceinline__ float row_max(float v) {
#pragma unroll
    for (int o = L / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

template <int DK, int DV>
struct Q8Io {
    static constexpr int LPR = DV / 4, RPP = 4 * DV / LPR, RPT = DK / RPP;
    // encode: m (the thread's float4 of rows rg + x*RPP) -> codes, scales
    // Row maxima and 127 / max of the thread's RPT rows.  With a warp per row (LPR = 32) the
    // 8 rows reduce in one butterfly that halves the rows a lane carries at every stage (9
    // shuffles instead of 40), lane groups of 4 then hold one row each and divide once per
    // row, and the results come back by shuffle; the values are the same as row by row.
    // my_x / my_scale: with LPR = 32, the row (index x) whose scale this lane stores (lanes with
    // lane % 4 == 0), else -1
    static __device__ __forceinline__ void row_stats(const float4 (&m)[RPT], int lane,
                                                     float (&amax)[RPT], float (&inv)[RPT],
                                                     int &my_x, float &my_scale) {
        my_x = -1;
        my_scale = 0.f;
        float v[RPT];
#pragma unroll
        for (int x = 0; x < RPT; ++x)
            v[x] = fmaxf(fmaxf(fabsf(m[x].x), fabsf(m[x].y)), fmaxf(fabsf(m[x].z), fabsf(m[x].w)));
        if constexpr (LPR == 32 && RPT == 8) {
            const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
            float w4[4], w2[2];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float send = b4 ? v[k] : v[k + 4], keep = b4 ? v[k + 4] : v[k];
                w4[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 16));
            }
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const float send = b3 ? w4[k] : w4[k + 2], keep = b3 ? w4[k + 2] : w4[k];
                w2[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 8));
            }
            float w1;
            {
                const float send = b2 ? w2[0] : w2[1], keep = b2 ? w2[1] : w2[0];
                w1 = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, 4));
            }
            w1 = fmaxf(w1, __shfl_xor_sync(0xffffffffu, w1, 2));
            w1 = fmaxf(w1, __shfl_xor_sync(0xffffffffu, w1, 1));
            // this lane now holds the max of row x = 4 b4 + 2 b3 + b2
            const float iv = w1 > 0.f ? __fdiv_rn(127.f, w1) : 0.f;
            if ((lane & 3) == 0) {
                my_x = (b4 ? 4 : 0) + (b3 ? 2 : 0) + (b2 ? 1 : 0);
                my_scale = w1 > 0.f ? __fdiv_rn(w1, 127.f) : 0.f;
            }
#pragma unroll
            for (int x = 0; x < RPT; ++x) {
                const int src = ((x >> 2) & 1) * 16 + ((x >> 1) & 1) * 8 + (x & 1) * 4;
                amax[x] = __shfl_sync(0xffffffffu, w1, src);
                inv[x] = __shfl_sync(0xffffffffu, iv, src);
            }
        } else {
#pragma unroll
            for (int x = 0; x < RPT; ++x) {
                amax[x] = row_max<LPR>(v[x]);
                float iv = 0.f;   // divided once per row and broadcast from its first lane
                if (lane % LPR == 0 && amax[x] > 0.f) iv = __fdiv_rn(127.f, amax[x]);
                inv[x] = __shfl_sync(0xffffffffu, iv, lane & ~(LPR - 1));
            }
        }
    }
    // Encode x = m (+ the residual e_in, error feedback) into codes and row scales.  Every code
    // draws its own dither u = (pcg_hash(index ^ hf) >> 8) * 2^-24, index = base_idx + row*DV + col.
    // With EF the new residual bf16(x - code*scale) goes to e_out (global, same layout as codes);
    // e_in is the previous residual (bf16, shared memory, same layout).
    template <bool EF = false>
    static __device__ __forceinline__ void store(float4 (&m)[RPT], int8_t *codes, float *scales,
                                                 uint32_t hf, uint32_t base_idx, int rg, int c4,
                                                 int lane, const __nv_bfloat16 *e_in = nullptr,
                                                 __nv_bfloat16 *e_out = nullptr) {
        if (EF && e_in) {   // (a null e_in: the first encode, residual zero)
#pragma unroll
            for (int x = 0; x < RPT; ++x) {
                const uint2 eb = *reinterpret_cast<const uint2 *>(e_in + (rg + x * RPP) * DV + c4);
                const float2 e01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&eb.x));
                const float2 e23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&eb.y));
                m[x].x = __fadd_rn(m[x].x, e01.x); m[x].y = __fadd_rn(m[x].y, e01.y);
                m[x].z = __fadd_rn(m[x].z, e23.x); m[x].w = __fadd_rn(m[x].w, e23.y);
            }
        }
        float amaxs[RPT], invs[RPT], my_scale;
        int my_x;
        row_stats(m, lane, amaxs, invs, my_x, my_scale);
        if constexpr (LPR == 32 && RPT == 8) {
            if (my_x >= 0) scales[rg + my_x * RPP] = my_scale;
        }
        // The hashed values of a thread's four codes are (idx0 + e) ^ hf with idx0 a multiple of 4
        // (so is c4): (idx0 ^ (hf & ~3)) + ((hf & 3) ^ e), the two terms sharing no bit.  The
        // hash's state, that value times 747796405 plus 2891336453 (mod 2^32), is then a per-row
        // product plus one of four per-call constants.
        uint32_t kst[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) kst[e] = ((hf & 3u) ^ (uint32_t)e) * 747796405u + 2891336453u;
#pragma unroll
        for (int x = 0; x < RPT; ++x) {
            const int row = rg + x * RPP;
            const float amax = amaxs[x], inv = invs[x];
            const float v[4] = {m[x].x, m[x].y, m[x].z, m[x].w};
            const uint32_t sb = ((base_idx + (uint32_t)(row * DV + c4)) ^ (hf & ~3u)) * 747796405u;
            int qq[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                // u = (r >> 8) * 2^-24, formed as (r with its low 8 bits cleared) * 2^-32: the same
                // value (at most 24 significant bits, exact in fp32), and the mask fuses with the
                // hash's last xor
                const uint32_t r = pcg_output(sb + kst[e]);   // == pcg_hash((idx0 + e) ^ hf)
                const float u = __fmul_rn(__uint2float_rn(r & 0xFFFFFF00u), 0x1p-32f);
                // a zero row has inv == 0, so its codes come out as floor(u) == 0 here too
                qq[e] = max(__float2int_rd(__fadd_rn(__fmul_rn(v[e], inv), u)), -127);
            }
            // the four codes into one word, the upper clamp at 127 done by the saturating pack:
            // bytes (q0, q1, q2, q3) from the low end
            uint32_t w32, hi16;
            asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, 0;" : "=r"(hi16) : "r"(qq[3]), "r"(qq[2]));
            asm("cvt.pack.sat.s8.s32.b32 %0, %1, %2, %3;" : "=r"(w32) : "r"(qq[1]), "r"(qq[0]), "r"(hi16));
            *reinterpret_cast<uint32_t *>(codes + row * DV + c4) = w32;
            if constexpr (!(LPR == 32 && RPT == 8))
                if (lane % LPR == 0) scales[row] = amax > 0.f ? __fdiv_rn(amax, 127.f) : 0.f;
            if constexpr (EF) {
                // the residual left for the next encode: bf16(x - code * scale), scale = amax / 127
                const float sc = amax > 0.f ? __fdiv_rn(amax, 127.f) : 0.f;
                float ev[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) ev[e] = __fsub_rn(v[e], __fmul_rn((float)min(qq[e], 127), sc));
                __nv_bfloat162 lo2 = __floats2bfloat162_rn(ev[0], ev[1]), hi2 = __floats2bfloat162_rn(ev[2], ev[3]);
                uint2 ob;
                ob.x = *reinterpret_cast<const uint32_t *>(&lo2);
                ob.y = *reinterpret_cast<const uint32_t *>(&hi2);
                *reinterpret_cast<uint2 *>(e_out + row * DV + c4) = ob;
            }
        }
    }
    // decode: codes, scales -> m
    static __device__ __forceinline__ void load(float4 (&m)[RPT], const int8_t *codes, const float *scales,
                                                int rg, int c4) {
#pragma unroll
        for (int x = 0; x < RPT; ++x) {
            const int row = rg + x * RPP;
            const char4 c = *reinterpret_cast<const char4 *>(codes + row * DV + c4);
            const float s = scales[row];
            // code c as a float by the conversion unit (the integer logic pipe is the busy one)
            auto cf = [](signed char v) { return __int2float_rn((int)v); };
            m[x] = make_float4(__fmul_rn(cf(c.x), s), __fmul_rn(cf(c.y), s), __fmul_rn(cf(c.z), s),
                               __fmul_rn(cf(c.w), s));
        }
    }
};

template <int DK, int DV, bool Q8 = false, bool EF = false>
struct StreamCfg {
    static constexpr int NT = 4 * DV;
    static constexpr int LPR = DV / 4, RPP = NT / LPR, RPT = DK / RPP;
    // bytes of one head state: fp32 M, or int8 codes followed by the fp32 row scales (and, with
    // error feedback, the bf16 residual)
    static constexpr int SLOT = Q8 ? DK * DV + DK * 4 + (EF ? DK * DV * 2 : 0) : DK * DV * 4;
    static constexpr int NS = SLOT >= 40960 ? 3 : (SLOT >= 16384 ? 8 : 16);
    static constexpr int CHUNK = SLOT < 16384 ? SLOT : 16384;       // bytes per bulk copy
    static constexpr int HB = 4;                                    // heads per record batch
    // largest (HB/G) * record size over G in {1, 2, 4}: the records of one batch
    static constexpr int rec_floats(int g) { return (2 * DK + 2 * g * DV + 2 * g + 2 + 3) & ~3; }
    static constexpr int max2(int x, int y) { return x > y ? x : y; }
    static constexpr int RECBUF = max2(max2(HB * rec_floats(1), (HB / 2) * rec_floats(2)), rec_floats(4));
};

// Every array read or written as float4 is 16-byte aligned explicitly.
template <int DK, int DV, bool Q8 = false, bool EF = false>
struct StreamTail {
    alignas(16) uint64_t full[StreamCfg<DK, DV, Q8, EF>::NS];
    alignas(16) uint64_t rfull[2];
    alignas(16) float rec[2][StreamCfg<DK, DV, Q8, EF>::RECBUF];   // records of the current / next batch
    alignas(16) float red_p[StreamCfg<DK, DV, Q8, EF>::RPP][DV];
    alignas(16) float red_s[StreamCfg<DK, DV, Q8, EF>::RPP][DV];
    alignas(16) float up[DV];
    alignas(16) float nw[DV];
    float npart[4];
    int rec_bad;
    int dead;      // a state wait gave up: every later item is handled like a padding lane
};

template <int DK, int DV, bool Q8 = false, bool EF = false>
constexpr size_t stream_smem_bytes() {
    return (size_t)StreamCfg<DK, DV, Q8, EF>::NS * StreamCfg<DK, DV, Q8, EF>::SLOT +
           sizeof(StreamTail<DK, DV, Q8, EF>);
}

__device__ __forceinline__ void named_bar(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

template <int DK, int DV, typename TOut, bool Q8 = false, bool EF = false>
__global__ void __launch_bounds__(4 * DV, 1) decode_stream_kernel(DecodeArgs a) {
    using Cfg = StreamCfg<DK, DV, Q8, EF>;
    constexpr int NT = Cfg::NT, LPR = Cfg::LPR, RPP = Cfg::RPP, RPT = Cfg::RPT, NS = Cfg::NS;
    constexpr int HB = Cfg::HB;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float *slots = reinterpret_cast<float *>(smem_raw);
    StreamTail<DK, DV, Q8, EF> &tl = *reinterpret_cast<StreamTail<DK, DV, Q8, EF> *>(smem_raw + NS * Cfg::SLOT);

    const Dims &d = a.d;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = d.grp;                 // 1, 2 or 4: HB % G == 0
    const DecRec R(DK, DV, G);
    const int n_units = a.n * d.hk;
    if ((int)blockIdx.x >= n_units) return;
    const int my_units = (n_units - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
    const int n_items = my_units * G;
    const int nub = HB / G;              // units per batch
    const int n_batches = (n_items + HB - 1) / HB;
    TOut *out = (TOut *)a.out;
    const int rg = tid / LPR, c4 = (tid % LPR) * 4;
    const uint32_t hframe = Q8 ? pcg_hash(a.frame) : 0u;   // keys the Q8 rounding dither

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) tc::mbar_init(tc::smem_u32(&tl.full[s]), 1);
        for (int s = 0; s < 2; ++s) tc::mbar_init(tc::smem_u32(&tl.rfull[s]), 1);
        tc::mbar_fence_init();
        tl.rec_bad = 0;
        tl.dead = 0;
    }
    for (int j = tid; j < DV; j += NT) tl.nw[j] = a.norm_w[j];
    __syncthreads();

    // producer (thread 0): bulk-load item `it`'s head state into slot it % NS
    auto issue = [&](int it) {
        const int u = (int)blockIdx.x + (it / G) * (int)gridDim.x, gi = it % G;
        const int n = u / d.hk, kh = u % d.hk;
        const int slot = a.state_idx ? a.state_idx[n] : n;
        const uint32_t mb = tc::smem_u32(&tl.full[it % NS]);
        if (slot < 0 || slot >= d.n_slots) {  // padding lane: complete the phase, no copy
            tc::mbar_arrive(mb);
            return;
        }
        if (it == 0 && blockIdx.x == 0 && (d.lose & LOSE_DECODE_STATE_COPY)) return;   // (tests)
        const long long head = (long long)slot * d.hv + (long long)kh * G + gi;
        const uint32_t dst = tc::smem_u32(slots) + (uint32_t)((it % NS) * Cfg::SLOT);
        tc::mbar_arrive_expect_tx(mb, Cfg::SLOT);
        if constexpr (Q8) {   // the codes, then the row scales (then the residual)
            tc::bulk_g2s(dst, a.q8 + head * DK * DV, DK * DV, mb);
            tc::bulk_g2s(dst + DK * DV, a.q8_scale + head * DK, DK * 4, mb);
            if constexpr (EF)
                tc::bulk_g2s(dst + DK * DV + DK * 4, a.q8_res + head * DK * DV, DK * DV * 2, mb);
        } else {
            const char *src = reinterpret_cast<const char *>(a.state + head * DK * DV);
            for (int c = 0; c < Cfg::SLOT; c += Cfg::CHUNK) tc::bulk_g2s(dst + c, src + c, Cfg::CHUNK, mb);
        }
    };
    // producer (thread 0): bulk-load the records of batch bb into buffer bb & 1
    auto issue_rec = [&](int bb) {
        if (bb >= n_batches) return;
        const uint32_t mb = tc::smem_u32(&tl.rfull[bb & 1]);
        int cnt = 0;
        for (int k = 0; k < nub; ++k) cnt += (bb * nub + k < my_units) ? 1 : 0;
        tc::mbar_arrive_expect_tx(mb, (uint32_t)(cnt * R.size * 4));
        for (int k = 0; k < nub; ++k) {
            const int uu = bb * nub + k;
            if (uu >= my_units) break;
            const int u = (int)blockIdx.x + uu * (int)gridDim.x;
            tc::bulk_g2s(tc::smem_u32(&tl.rec[bb & 1][k * R.size]), a.ws + (long long)u * R.size,
                         (uint32_t)(R.size * 4), mb);
        }
    };
    // The state ring does not depend on the prep kernel: start it, then wait
    // for the prep grid (a no-op when launched without programmatic
    // serialisation) before the first record copy.
    int n_issued = 0;   // (thread 0) items whose state copy has been issued
    if (tid == 0)
        for (; n_issued < NS && n_issued < n_items; ++n_issued) issue(n_issued);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (tid == 0) issue_rec(0);
    const uint64_t WL = d.wait_ns;

    for (int it = 0; it < n_items; ++it) {
        const int hb = it % HB, bb = it / HB;
        if (hb == 0) {
            // Thread 0 refills the other record buffer (every thread is done with
            // batch bb-1's records) and waits for this batch's; a wait that gives
            // up marks every later record bad, for all threads alike.
            __syncthreads();
            if (tid == 0) {
                tc::fence_async_smem();
                issue_rec(bb + 1);
                if (!tl.rec_bad && !tc::mbar_wait(tc::smem_u32(&tl.rfull[bb & 1]), (uint32_t)((bb >> 1) & 1), WL)) {
                    tl.rec_bad = 1;
                    set_error(a.err, GDN_DEVERR_TIMEOUT);
                }
            }
            __syncthreads();
        }
        const int ub = hb / G, gi = it % G;
        const float *rc = &tl.rec[bb & 1][ub * R.size];
        const int u = (int)blockIdx.x + (it / G) * (int)gridDim.x;
        const int n = u / d.hk, kh = u % d.hk, h = kh * G + gi;
        const long long out_row = (long long)n * d.hv * DV;
        const int rslot = __float_as_int(rc[R.slot]);
        int slot = (tl.rec_bad || rslot >= d.n_slots) ? -1 : rslot;
        // ---- this head's state has arrived?  A wait that gives up marks the CTA dead; from
        // the barrier below on, every thread treats this and every later item as a padding
        // lane (no state store), and no further copy is issued.
        bool here = slot >= 0 && !tl.dead;
        if (here && !tc::mbar_wait(tc::smem_u32(&tl.full[it % NS]), (uint32_t)((it / NS) & 1), WL)) {
            here = false;
            tl.dead = 1;
            set_error(a.err, GDN_DEVERR_TIMEOUT);
        }
        const unsigned char *Sb = reinterpret_cast<const unsigned char *>(slots) + (it % NS) * Cfg::SLOT;
        float4 m[RPT];
        float kr[RPT];
        if (here) {
            float qr[RPT];
            if constexpr (Q8) {
                Q8Io<DK, DV>::load(m, reinterpret_cast<const int8_t *>(Sb),
                                   reinterpret_cast<const float *>(Sb + DK * DV), rg, c4);
            } else {
#pragma unroll
                for (int x = 0; x < RPT; ++x)
                    m[x] = *reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(Sb) +
                                                             (rg + x * RPP) * DV + c4);
            }
#pragma unroll
            for (int x = 0; x < RPT; ++x) {
                kr[x] = rc[R.k + rg + x * RPP];
                qr[x] = rc[R.q + rg + x * RPP];
            }
            float4 pp = make_float4(0.f, 0.f, 0.f, 0.f), ss = pp;
#pragma unroll
            for (int x = 0; x < RPT; ++x) {
                pp.x += m[x].x * kr[x]; pp.y += m[x].y * kr[x]; pp.z += m[x].z * kr[x]; pp.w += m[x].w * kr[x];
                ss.x += m[x].x * qr[x]; ss.y += m[x].y * qr[x]; ss.z += m[x].z * qr[x]; ss.w += m[x].w * qr[x];
            }
            *reinterpret_cast<float4 *>(&tl.red_p[rg][c4]) = pp;
            *reinterpret_cast<float4 *>(&tl.red_s[rg][c4]) = ss;
        }
        __syncthreads();  // (A) every thread holds its part of the slot in registers
        if (tl.dead) slot = -1;
        if (tid == 0 && !tl.dead && it + NS < n_items) {
            tc::fence_async_smem();
            issue(it + NS);
            n_issued = it + NS + 1;
        }
        if (slot < 0) {   // padding lane: zero output row of this head
            for (int j = tid; j < DV; j += NT) out[out_row + (long long)h * DV + j] = from_f32<TOut>(0.f);
            continue;
        }
        const float ga = rc[R.ga + gi], gb = rc[R.gb + gi];
        float ov = 0.f;
        if (tid < DV) {
            float p = 0.f, s2 = 0.f;
#pragma unroll
            for (int r = 0; r < RPP; ++r) {
                p += tl.red_p[r][tid];
                s2 += tl.red_s[r][tid];
            }
            const float uu = gb * (rc[R.v + gi * DV + tid] - ga * p);
            tl.up[tid] = uu;
            ov = ga * s2 + uu * rc[R.kq];
        }
        __syncthreads();  // (B)
        {
            const long long head = (long long)slot * d.hv + h;
            const float4 u4 = *reinterpret_cast<const float4 *>(&tl.up[c4]);
#pragma unroll
            for (int x = 0; x < RPT; ++x) {
                m[x].x = ga * m[x].x + kr[x] * u4.x;
                m[x].y = ga * m[x].y + kr[x] * u4.y;
                m[x].z = ga * m[x].z + kr[x] * u4.z;
                m[x].w = ga * m[x].w + kr[x] * u4.w;
            }
            if constexpr (Q8) {
                Q8Io<DK, DV>::template store<EF>(
                    m, a.q8 + head * DK * DV, a.q8_scale + head * DK, hframe, (uint32_t)(head * DK * DV), rg,
                    c4, lane, reinterpret_cast<const __nv_bfloat16 *>(Sb + DK * DV + DK * 4),
                    EF ? a.q8_res + head * DK * DV : nullptr);
            } else {
                float *Mg = a.state + head * DK * DV;
#pragma unroll
                for (int x = 0; x < RPT; ++x)
                    *reinterpret_cast<float4 *>(Mg + (long long)(rg + x * RPP) * DV + c4) = m[x];
            }
        }
        if (tid < DV) {   // gated RMSNorm of this head's o, among the DV threads that hold it
            const float sq = warp_sum(ov * ov);
            if (lane == 0) tl.npart[warp] = sq;
            named_bar(1, DV);
            float tot = 0.f;
#pragma unroll
            for (int wi = 0; wi < DV / 32; ++wi) tot += tl.npart[wi];
            const float rs = rsqrtf(tot / (float)DV + d.norm_eps);
            out[out_row + (long long)h * DV + tid] =
                from_f32<TOut>(ov * rs * tl.nw[tid] * rc[R.z + gi * DV + tid]);
        }
    }
    // After a timeout, shared memory must outlive every copy still in flight: thread 0 waits
    // (bounded) for the state copies it issued and never consumed, and for the next batch of
    // records.  Without a timeout every issued copy has been waited for already.
    __syncthreads();
    if (tid == 0 && (tl.dead || tl.rec_bad)) {
        for (int j = n_issued - NS < 0 ? 0 : n_issued - NS; j < n_issued; ++j)
            tc::mbar_wait(tc::smem_u32(&tl.full[j % NS]), (uint32_t)((j / NS) & 1), WL);
        for (int b = 0; b < 2; ++b)
            tc::mbar_wait(tc::smem_u32(&tl.rfull[b]), 0u, WL), tc::mbar_wait(tc::smem_u32(&tl.rfull[b]), 1u, WL);
    }
}

template <int DK, int DV, typename TA, typename TOut, bool Q8 = false, bool EF = false>
static cudaError_t launch_stream_t(const DecodeArgs &a, cudaStream_t s) {
    const int units = a.n * a.d.hk;
    if (a.d.grp == 1) decode_prep_kernel<DK, DV, TA, 1><<<units, 256, 0, s>>>(a);
    else if (a.d.grp == 2) decode_prep_kernel<DK, DV, TA, 2><<<units, 256, 0, s>>>(a);
    else decode_prep_kernel<DK, DV, TA, 4><<<units, 256, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    auto kern = decode_stream_kernel<DK, DV, TOut, Q8, EF>;
    constexpr size_t smem = stream_smem_bytes<DK, DV, Q8, EF>();
    static_assert(smem <= 227 * 1024, "the state ring and its tail exceed one CTA's shared memory");
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // programmatic dependent launch: overlaps this kernel's launch and its
    // first state copies with the tail of the prep kernel
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(units < sm_count() ? units : sm_count());
    lc.blockDim = dim3(4 * DV);
    lc.dynamicSmemBytes = smem;
    lc.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    lc.attrs = at;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, kern, a);
}

template <int DK, int DV, typename TA, typename TOut>
static cudaError_t launch_dec_t(const DecodeArgs &a, bool fused, cudaStream_t s) {
    dim3 grid(a.n * a.d.hk);
    if (fused)
        return launch_stream_t<DK, DV, TA, TOut>(a, s);
    else
        decode_kernel<DK, DV, TA, TOut><<<grid, 4 * DV, 0, s>>>(a);
    return cudaGetLastError();
}

template <int DK, int DV>
static cudaError_t launch_dec_d(const DecodeArgs &a, bool fused, bool in_bf16, bool out_bf16,
                                cudaStream_t s) {
    if (in_bf16)
        return out_bf16 ? launch_dec_t<DK, DV, __nv_bfloat16, __nv_bfloat16>(a, fused, s)
                        : launch_dec_t<DK, DV, __nv_bfloat16, float>(a, fused, s);
    return out_bf16 ? launch_dec_t<DK, DV, float, __nv_bfloat16>(a, fused, s)
                    : launch_dec_t<DK, DV, float, float>(a, fused, s);
}

cudaError_t launch_decode(const DecodeArgs &a, bool fused, bool in_bf16, bool out_bf16,
                          cudaStream_t s) {
    if (a.n == 0) return cudaSuccess;
    if (a.d.grp > DecodeCfg<32, 32>::MAXG) return cudaErrorInvalidValue;
    switch (a.d.dk) {
        case 32: return launch_dec_d<32, 32>(a, fused, in_bf16, out_bf16, s);
        case 64: return launch_dec_d<64, 64>(a, fused, in_bf16, out_bf16, s);
        case 128: return launch_dec_d<128, 128>(a, fused, in_bf16, out_bf16, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn

namespace gdn {
size_t decode_ws_bytes(const Dims &d, long long n_seqs) {
    const DecRec R(d.dk, d.dv, d.grp);
    return (size_t)(n_seqs > 0 ? n_seqs : 0) * d.hk * R.size * sizeof(float);
}
}  // namespace gdn

// ---------------------------------------------------------------------------
// Q8 recurrent state (int8 codes + one fp32 scale per state row), the decode
// variant that cuts the state bytes about 4x.  Row i of a head's M (dv
// values) is stored as code_ij * s_i with s_i = max_j |M_ij| / 127; a new
// state is encoded with stochastic rounding, code = floor(M * 127/max + u),
// u in [0, 1) from a counter-based hash of (frame, slot, head, i, j), so that
// the rounding error has zero mean and does not accumulate a bias across
// steps.  The hash is the PCG hash of Jarzynski and Olano ("Hash Functions for
// GPU Rendering", JCGT 2020): one PCG32 LCG step and its RXS-M-XS output.
// Every step of the encoding is an explicitly rounded fp32 operation.
namespace gdn {

namespace {

// fp32 pool <-> Q8 pool, one CTA per (slot, head)
// (to Q8 with a residual pool: the first encode of an error-feedback pool, residual in = 0)
template <int DK, int DV>
__global__ void __launch_bounds__(4 * DV) q8_convert_kernel(Dims d, const float *state, int8_t *codes,
                                                            float *scales, __nv_bfloat16 *res,
                                                            uint32_t frame, bool to_q8) {
    using Q = Q8Io<DK, DV>;
    const int tid = threadIdx.x, lane = tid & 31;
    const long long head = blockIdx.x;                       // slot * HV + h
    const int rg = tid / Q::LPR, c4 = (tid % Q::LPR) * 4;
    int8_t *cp = codes + head * DK * DV;
    float *sp = scales + head * DK;
    float4 m[Q::RPT];
    if (to_q8) {
#pragma unroll
        for (int x = 0; x < Q::RPT; ++x)
            m[x] = *reinterpret_cast<const float4 *>(state + head * DK * DV + (rg + x * Q::RPP) * DV + c4);
        if (res) {
            Q::template store<true>(m, cp, sp, pcg_hash(frame), (uint32_t)(head * DK * DV), rg, c4, lane,
                                    nullptr, res + head * DK * DV);
        } else {
            Q::store(m, cp, sp, pcg_hash(frame), (uint32_t)(head * DK * DV), rg, c4, lane);
        }
    } else {
        Q::load(m, cp, sp, rg, c4);
        float *out = const_cast<float *>(state);
#pragma unroll
        for (int x = 0; x < Q::RPT; ++x)
            *reinterpret_cast<float4 *>(out + head * DK * DV + (rg + x * Q::RPP) * DV + c4) = m[x];
    }
}

template <int D, typename TA, typename TOut>
cudaError_t launch_q8_t(const DecodeArgs &a, cudaStream_t s) {
    // prep + the streaming kernel on Q8 slots (with the residual when error feedback is on)
    return a.q8_res ? launch_stream_t<D, D, TA, TOut, true, true>(a, s)
                    : launch_stream_t<D, D, TA, TOut, true, false>(a, s);
}

template <int D>
cudaError_t launch_q8_d(const DecodeArgs &a, bool in_bf16, bool out_bf16, cudaStream_t s) {
    if (in_bf16)
        return out_bf16 ? launch_q8_t<D, __nv_bfloat16, __nv_bfloat16>(a, s)
                        : launch_q8_t<D, __nv_bfloat16, float>(a, s);
    return out_bf16 ? launch_q8_t<D, float, __nv_bfloat16>(a, s) : launch_q8_t<D, float, float>(a, s);
}

}  // namespace

cudaError_t launch_decode_q8(const DecodeArgs &a, bool in_bf16, bool out_bf16, cudaStream_t s) {
    if (a.n == 0) return cudaSuccess;
    if (a.d.grp > 4 || !a.q8 || !a.q8_scale) return cudaErrorInvalidValue;
    switch (a.d.dk) {
        case 32: return launch_q8_d<32>(a, in_bf16, out_bf16, s);
        case 64: return launch_q8_d<64>(a, in_bf16, out_bf16, s);
        case 128: return launch_q8_d<128>(a, in_bf16, out_bf16, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_q8_convert(const Dims &d, const float *state, int8_t *codes, float *scales,
                              __nv_bfloat16 *res, uint32_t frame, bool to_q8, cudaStream_t s) {
    const long long heads = (long long)d.n_slots * d.hv;
    if (heads == 0) return cudaSuccess;
    switch (d.dk) {
        case 32: q8_convert_kernel<32, 32><<<(unsigned)heads, 128, 0, s>>>(d, state, codes, scales, res, frame, to_q8); break;
        case 64: q8_convert_kernel<64, 64><<<(unsigned)heads, 256, 0, s>>>(d, state, codes, scales, res, frame, to_q8); break;
        case 128: q8_convert_kernel<128, 128><<<(unsigned)heads, 512, 0, s>>>(d, state, codes, scales, res, frame, to_q8); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace gdn
