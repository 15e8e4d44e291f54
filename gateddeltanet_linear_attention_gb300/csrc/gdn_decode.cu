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
// The fused form also runs, for the same CTA, the conv step of the q/k
// channels of its q/k head and the v channels of its v-heads (each history
// has exactly one owner, so the in-place shift is race-free), SiLU, the q/k L2
// norm, the gates and the gated RMSNorm: one launch per decode step.
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

template <int DK, int DV, typename TA, typename TOut, bool FUSED>
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
    if (FUSED) {
        const TA *x = (const TA *)a.x + (long long)n * a.ld_x;
        const TA *w = (const TA *)a.conv_w;
        TA *cs = (TA *)a.conv_state + (long long)slot * d.ch * 3;
        const int nch = 2 * DK + G * DV;
        for (int ci = tid; ci < nch; ci += NT) {
            int c;
            if (ci < DK) c = kh * DK + ci;
            else if (ci < 2 * DK) c = d.hk * DK + kh * DK + (ci - DK);
            else c = 2 * d.hk * DK + kh * G * DV + (ci - 2 * DK);
            TA *hc = cs + (long long)c * 3;
            TA h0 = hc[0], h1 = hc[1], h2 = hc[2], xc = x[c];
            float acc = to_f32(w[c * 4 + 0]) * to_f32(h0) + to_f32(w[c * 4 + 1]) * to_f32(h1) +
                        to_f32(w[c * 4 + 2]) * to_f32(h2) + to_f32(w[c * 4 + 3]) * to_f32(xc);
            hc[0] = h1;
            hc[1] = h2;
            hc[2] = xc;
            float val = silu_f(acc);
            if (ci < DK) qs[ci] = val;
            else if (ci < 2 * DK) ks[ci - DK] = val;
            else vs[(ci - 2 * DK) / DV][(ci - 2 * DK) % DV] = val;
        }
        if (tid < G) {
            const int h = kh * G + tid;
            const TA *u = (const TA *)a.u + (long long)n * a.ld_ub;
            const TA *b = (const TA *)a.b_logit + (long long)n * a.ld_ub;
            float gg = -expf(a.A_log[h]) * softplus_f(to_f32(u[h]) + a.dt_bias[h]);
            gate_a[tid] = expf(gg);
            gate_b[tid] = sigmoid_f(to_f32(b[h]));
        }
    } else {
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
    const bool l2 = FUSED || (a.flags & GDN_FLAG_L2NORM_QK);
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
        if (FUSED) {
            float ov = tid < DV ? os[tid] : 0.f;
            float sq = warp_sum(ov * ov);
            if (tid < DV && lane == 0) red_p[0][warp] = sq;  // red_p is free again here
            __syncthreads();
            if (tid < DV) {
                float tot = 0.f;
                for (int wi = 0; wi < DV / 32; ++wi) tot += red_p[0][wi];
                float rs = rsqrtf(tot / (float)DV + d.norm_eps);
                const TA *z = (const TA *)a.z + (long long)n * a.ld_z + (long long)h * DV;
                out[out_row + (long long)h * DV + tid] =
                    from_f32<TOut>(ov * rs * a.norm_w[tid] * silu_f(to_f32(z[tid])));
            }
        } else {
            if (tid < DV) out[out_row + (long long)h * DV + tid] = from_f32<TOut>(os[tid]);
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Streaming form of the fused decode (the product path).  A persistent grid of
// one CTA per SM walks its (sequence, q/k head) units; each unit's G head
// states (dk*dv*4 bytes each) flow HBM -> shared memory through a ring of NS
// slots filled by bulk asynchronous copies (cp.async.bulk, completion counted
// on one mbarrier per slot), so that while one head is being updated the next
// NS-1 are already in flight.  The small per-unit inputs (conv step of the
// unit's q/k/v channels, SiLU, L2, gates, and the z rows of the norm) are
// computed for a batch of HB heads at once, so their global loads overlap
// each other and the state copies instead of sitting on every head's critical
// path; per head only shared memory is touched before the state write.
template <int DK, int DV>
struct StreamCfg {
    static constexpr int NT = 4 * DV;
    static constexpr int LPR = DV / 4, RPP = NT / LPR, RPT = DK / RPP;
    static constexpr int SLOT = DK * DV * 4;                        // bytes of one head state
    static constexpr int NS = SLOT >= 65536 ? 3 : (SLOT >= 16384 ? 8 : 16);
    static constexpr int CHUNK = SLOT < 16384 ? SLOT : 16384;       // bytes per bulk copy
    static constexpr int HB = 4;                                    // heads per prologue batch
};

// Every array read or written as float4 is 16-byte aligned explicitly.
template <int DK, int DV>
struct StreamTail {
    static constexpr int HB = StreamCfg<DK, DV>::HB;
    alignas(16) uint64_t full[StreamCfg<DK, DV>::NS];
    alignas(16) float qk[HB][2][DK];      // normalised q (0) and k (1) per unit of the batch
    alignas(16) float vs[HB][DV];         // conv'd v per head of the batch
    alignas(16) float zs[HB][DV];         // SiLU(z) per head of the batch
    alignas(16) float red_p[StreamCfg<DK, DV>::RPP][DV];
    alignas(16) float red_s[StreamCfg<DK, DV>::RPP][DV];
    alignas(16) float up[DV];
    alignas(16) float nw[DV];
    float gate_a[HB], gate_b[HB];
    float ssq[HB][2];                     // |q|^2, |k|^2 per unit
    float kq[HB];
    float npart[4];
    int uslot[HB];
};

template <int DK, int DV>
constexpr size_t stream_smem_bytes() {
    return (size_t)StreamCfg<DK, DV>::NS * StreamCfg<DK, DV>::SLOT + sizeof(StreamTail<DK, DV>);
}

__device__ __forceinline__ void named_bar(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

template <int DK, int DV, typename TA, typename TOut>
__global__ void __launch_bounds__(4 * DV, 1) decode_stream_kernel(DecodeArgs a) {
    using Cfg = StreamCfg<DK, DV>;
    constexpr int NT = Cfg::NT, LPR = Cfg::LPR, RPP = Cfg::RPP, RPT = Cfg::RPT, NS = Cfg::NS;
    constexpr int HB = Cfg::HB;
    extern __shared__ __align__(128) unsigned char smem_raw[];
    float *slots = reinterpret_cast<float *>(smem_raw);
    StreamTail<DK, DV> &tl = *reinterpret_cast<StreamTail<DK, DV> *>(smem_raw + NS * Cfg::SLOT);

    const Dims &d = a.d;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = d.grp;                 // 1, 2 or 4: HB % G == 0
    const int n_units = a.n * d.hk;
    if ((int)blockIdx.x >= n_units) return;
    const int my_units = (n_units - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x;
    const int n_items = my_units * G;
    TOut *out = (TOut *)a.out;
    const int rg = tid / LPR, c4 = (tid % LPR) * 4;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) tc::mbar_init(tc::smem_u32(&tl.full[s]), 1);
        tc::mbar_fence_init();
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
        const char *src = reinterpret_cast<const char *>(
            a.state + ((long long)slot * d.hv + (long long)kh * G + gi) * DK * DV);
        const uint32_t dst = tc::smem_u32(slots) + (uint32_t)((it % NS) * Cfg::SLOT);
        tc::mbar_arrive_expect_tx(mb, Cfg::SLOT);
        for (int c = 0; c < Cfg::SLOT; c += Cfg::CHUNK) tc::bulk_g2s(dst + c, src + c, Cfg::CHUNK, mb);
    };
    if (tid == 0)
        for (int it = 0; it < NS && it < n_items; ++it) issue(it);

    bool timed_out = false;
    for (int it = 0; it < n_items; ++it) {
        const int hb = it % HB;
        if (hb == 0) {
            // ---- batch prologue for heads it .. it+HB-1 (units it/G .. (it+HB-1)/G)
            __syncthreads();   // the previous batch's inputs are no longer read
            const int ub0 = it / G, nub = HB / G;
            const int nch = 2 * DK + G * DV;
            for (int idx = tid; idx < nub * nch; idx += NT) {
                const int ub = idx / nch, ci = idx % nch;
                const int uu = ub0 + ub;
                if (uu >= my_units) continue;
                const int u = (int)blockIdx.x + uu * (int)gridDim.x;
                const int n = u / d.hk, kh = u % d.hk;
                const int slot = a.state_idx ? a.state_idx[n] : n;
                if (slot < 0 || slot >= d.n_slots) continue;
                int c;
                if (ci < DK) c = kh * DK + ci;
                else if (ci < 2 * DK) c = d.hk * DK + kh * DK + (ci - DK);
                else c = 2 * d.hk * DK + kh * G * DV + (ci - 2 * DK);
                const TA *x = (const TA *)a.x + (long long)n * a.ld_x;
                const TA *w = (const TA *)a.conv_w;
                TA *hc = (TA *)a.conv_state + ((long long)slot * d.ch + c) * 3;
                TA h0 = hc[0], h1 = hc[1], h2 = hc[2], xc = x[c];
                float acc = to_f32(w[c * 4 + 0]) * to_f32(h0) + to_f32(w[c * 4 + 1]) * to_f32(h1) +
                            to_f32(w[c * 4 + 2]) * to_f32(h2) + to_f32(w[c * 4 + 3]) * to_f32(xc);
                hc[0] = h1;
                hc[1] = h2;
                hc[2] = xc;
                const float val = silu_f(acc);
                if (ci < 2 * DK) tl.qk[ub][ci / DK][ci % DK] = val;
                else tl.vs[ub * G + (ci - 2 * DK) / DV][(ci - 2 * DK) % DV] = val;
            }
            for (int idx = tid; idx < HB * DV; idx += NT) {   // SiLU(z) of the batch's heads
                const int hbi = idx / DV, j = idx % DV;
                const int uu = ub0 + hbi / G;
                if (uu >= my_units) continue;
                const int u = (int)blockIdx.x + uu * (int)gridDim.x;
                const int n = u / d.hk, h = (u % d.hk) * G + hbi % G;
                const TA *z = (const TA *)a.z + (long long)n * a.ld_z + (long long)h * DV;
                tl.zs[hbi][j] = silu_f(to_f32(z[j]));
            }
            if (tid < HB) {
                const int uu = ub0 + tid / G;
                float ga = 0.f, gb = 0.f;
                if (uu < my_units) {
                    const int u = (int)blockIdx.x + uu * (int)gridDim.x;
                    const int n = u / d.hk, h = (u % d.hk) * G + tid % G;
                    const TA *uv = (const TA *)a.u + (long long)n * a.ld_ub;
                    const TA *bv = (const TA *)a.b_logit + (long long)n * a.ld_ub;
                    const float gg = -expf(a.A_log[h]) * softplus_f(to_f32(uv[h]) + a.dt_bias[h]);
                    ga = expf(gg);
                    gb = sigmoid_f(to_f32(bv[h]));
                }
                tl.gate_a[tid] = ga;
                tl.gate_b[tid] = gb;
            }
            if (tid < nub) {
                const int uu = ub0 + tid;
                int slot = -1;
                if (uu < my_units) {
                    const int u = (int)blockIdx.x + uu * (int)gridDim.x;
                    slot = slot_of(a.state_idx, u / d.hk, d.n_slots, a.err);
                }
                tl.uslot[tid] = slot;
            }
            __syncthreads();
            if (warp < 2 * nub) {    // |q|^2 and |k|^2 of each unit, one warp per vector
                const float *vec = tl.qk[warp >> 1][warp & 1];
                float ss = 0.f;
                for (int i = lane; i < DK; i += 32) ss += vec[i] * vec[i];
                ss = warp_sum(ss);
                if (lane == 0) tl.ssq[warp >> 1][warp & 1] = ss;
            }
            __syncthreads();
            for (int idx = tid; idx < nub * 2 * DK; idx += NT) {
                const int ub = idx / (2 * DK), part = (idx / DK) & 1, i = idx % DK;
                float f = rsqrtf(tl.ssq[ub][part] + d.l2_eps);
                if (part == 0) f *= d.q_scale;
                tl.qk[ub][part][i] *= f;
            }
            __syncthreads();
            if (warp < nub) {
                float kq = 0.f;
                for (int i = lane; i < DK; i += 32) kq += tl.qk[warp][0][i] * tl.qk[warp][1][i];
                kq = warp_sum(kq);
                if (lane == 0) tl.kq[warp] = kq;
            }
            __syncthreads();
        }
        const int ub = hb / G, gi = it % G;
        const int u = (int)blockIdx.x + (it / G) * (int)gridDim.x;
        const int n = u / d.hk, kh = u % d.hk, h = kh * G + gi;
        const long long out_row = (long long)n * d.hv * DV;
        const int slot = tl.uslot[ub];
        // ---- this head's state has arrived?
        if (!timed_out && !tc::mbar_wait(tc::smem_u32(&tl.full[it % NS]), (uint32_t)((it / NS) & 1))) {
            timed_out = true;
            set_error(a.err, GDN_DEVERR_TIMEOUT);
        }
        const float *Ms = slots + (it % NS) * (DK * DV);
        float4 m[RPT];
        float kr[RPT];
        if (slot >= 0) {
            float qr[RPT];
#pragma unroll
            for (int x = 0; x < RPT; ++x) {
                m[x] = *reinterpret_cast<const float4 *>(Ms + (rg + x * RPP) * DV + c4);
                kr[x] = tl.qk[ub][1][rg + x * RPP];
                qr[x] = tl.qk[ub][0][rg + x * RPP];
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
        if (tid == 0 && it + NS < n_items) {
            tc::fence_async_smem();
            issue(it + NS);
        }
        if (slot < 0) {   // padding lane: zero output row of this head
            for (int j = tid; j < DV; j += NT) out[out_row + (long long)h * DV + j] = from_f32<TOut>(0.f);
            continue;
        }
        const float ga = tl.gate_a[hb], gb = tl.gate_b[hb];
        float ov = 0.f;
        if (tid < DV) {
            float p = 0.f, s2 = 0.f;
#pragma unroll
            for (int r = 0; r < RPP; ++r) {
                p += tl.red_p[r][tid];
                s2 += tl.red_s[r][tid];
            }
            const float uu = gb * (tl.vs[hb][tid] - ga * p);
            tl.up[tid] = uu;
            ov = ga * s2 + uu * tl.kq[ub];
        }
        __syncthreads();  // (B)
        {
            float *Mg = a.state + ((long long)slot * d.hv + h) * DK * DV;
            const float4 u4 = *reinterpret_cast<const float4 *>(&tl.up[c4]);
#pragma unroll
            for (int x = 0; x < RPT; ++x) {
                float4 mn;
                mn.x = ga * m[x].x + kr[x] * u4.x;
                mn.y = ga * m[x].y + kr[x] * u4.y;
                mn.z = ga * m[x].z + kr[x] * u4.z;
                mn.w = ga * m[x].w + kr[x] * u4.w;
                *reinterpret_cast<float4 *>(Mg + (long long)(rg + x * RPP) * DV + c4) = mn;
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
            out[out_row + (long long)h * DV + tid] = from_f32<TOut>(ov * rs * tl.nw[tid] * tl.zs[hb][tid]);
        }
    }
}

template <int DK, int DV, typename TA, typename TOut>
static cudaError_t launch_stream_t(const DecodeArgs &a, cudaStream_t s) {
    auto kern = decode_stream_kernel<DK, DV, TA, TOut>;
    constexpr size_t smem = stream_smem_bytes<DK, DV>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int units = a.n * a.d.hk;
    const int grid = units < sm_count() ? units : sm_count();
    kern<<<grid, 4 * DV, smem, s>>>(a);
    return cudaGetLastError();
}

template <int DK, int DV, typename TA, typename TOut>
static cudaError_t launch_dec_t(const DecodeArgs &a, bool fused, cudaStream_t s) {
    dim3 grid(a.n * a.d.hk);
    if (fused)
        return launch_stream_t<DK, DV, TA, TOut>(a, s);
    else
        decode_kernel<DK, DV, TA, TOut, false><<<grid, 4 * DV, 0, s>>>(a);
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
