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
    __shared__ float qs[DK], ks[DK];
    __shared__ float vs[Cfg::MAXG][DV];
    __shared__ float gate_a[Cfg::MAXG], gate_b[Cfg::MAXG];
    __shared__ float red_p[RPP][DV], red_s[RPP][DV];
    __shared__ float up[DV], os[DV];
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

template <int DK, int DV, typename TA, typename TOut>
static cudaError_t launch_dec_t(const DecodeArgs &a, bool fused, cudaStream_t s) {
    dim3 grid(a.n * a.d.hk);
    if (fused)
        decode_kernel<DK, DV, TA, TOut, true><<<grid, 4 * DV, 0, s>>>(a);
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
