// gdn_verify.cu -- multi-token verification decode (hyperflare core-design,
// speculative target state: eight recurrent checkpoint columns per request, a
// round writes the columns of its verification inputs, and the committed
// column is the one of the last accepted input).
//
// For sequence n with k tokens t_0 .. t_{k-1} and source slot s, the
// one-token rule of gdn_decode.cu is applied k times in a row, starting from
// state and conv history of slot s (read only); after token j the state and
// the conv history (its last three raw inputs) are written to slot
// ckpt_idx[n] + j, and y_j is the gated-norm output of token j.
//
// One launch: verify_kernel, one CTA per (sequence, v-head), the G v-heads of
// a q/k head forming one thread-block cluster.  A CTA issues the loads of its
// head state (into registers: thread = one float4 column group of RPT rows)
// first; while they are in flight it runs the conv over the k tokens for the
// q and k channels of its q/k head and the v channels of its own head (one
// thread per channel; the other threads take SiLU(z) and the gates), the
// SiLU, the q/k L2 norms and k.q, into k records in shared memory.  The q/k
// channels are shared by the cluster's CTAs and each computes them itself;
// the first CTA of the cluster writes their checkpoint histories, after a
// cluster barrier that every CTA reaches only once its reads of the source
// history are done (a checkpoint column may be the source slot).  Then the
// state is carried through the k tokens and every token's state goes straight
// from registers to its column.  HBM bytes per head: (1 + k) * dk*dv*4.
#include "gdn_common.cuh"

namespace gdn {

namespace {

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

template <int DK, int DV, typename TA, typename TOut>
__global__ void __launch_bounds__(4 * DV, 2) verify_kernel(DecodeArgs a) {
    static_assert(DK == DV, "one thread per q, k and v channel, the last DV threads take z and the gates");
    constexpr int NT = 4 * DV, LPR = DV / 4, RPP = NT / LPR, RPT = DK / RPP, NW = NT / 32;
    extern __shared__ __align__(16) float recs[];   // the k records of this head
    __shared__ __align__(16) float red_p[RPP][DV];
    __shared__ __align__(16) float red_s[RPP][DV];
    __shared__ __align__(16) float up[DV];
    __shared__ float npart[DV / 32];
    __shared__ float nfac[2 * kMaxVerify];           // L2 factors: q of token j at 2j, k at 2j + 1
    const Dims &d = a.d;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = d.grp, K = a.k_tokens;
    const int n = blockIdx.x / d.hv, h = blockIdx.x % d.hv, kh = h / G, gi = h % G;
    const DecRec R(DK, DV, 1);
    TOut *out = (TOut *)a.out;
    // The slot, the columns and so the early exit are the same for every CTA of the cluster
    // (one sequence), so no CTA leaves while another waits at the cluster barrier.
    const bool lead = tid == 0 && gi == 0;
    const int slot = slot_of(a.state_idx, n, d.n_slots, lead ? a.err : nullptr);
    int ck = -1;
    if (slot >= 0) {
        ck = a.ckpt_idx[n];
        if (ck < 0 || ck + K > d.n_slots) {
            if (lead) set_error(a.err, GDN_DEVERR_SLOT);
            ck = -1;
        }
    }
    if (slot < 0 || ck < 0) {   // padding lane (or rejected columns): zero outputs, no state traffic
        for (int e = tid; e < K * DV; e += NT) {
            const int j = e / DV, idx = e % DV;
            out[(long long)(n * K + j) * d.hv * DV + (long long)h * DV + idx] = from_f32<TOut>(0.f);
        }
        return;
    }
    // ---- the head state: its loads go out first
    const int rg = tid / LPR, c4 = (tid % LPR) * 4;
    float4 m[RPT];
    {
        const float *Ms = a.state + ((long long)slot * d.hv + h) * DK * DV;
#pragma unroll
        for (int x = 0; x < RPT; ++x)
            m[x] = *reinterpret_cast<const float4 *>(Ms + (long long)(rg + x * RPP) * DV + c4);
    }
    // ---- the token inputs: thread t < 2 DK + DV owns one channel (q, k of the q/k head, v of
    // this head); thread 2 DK + DV + e owns column e of z and, for e < k, the gates of token e
    const TA *w = (const TA *)a.conv_w;
    const TA *src = (const TA *)a.conv_state + (long long)slot * d.ch * 3;
    TA *cols = (TA *)a.conv_state + (long long)ck * d.ch * 3;
    const long long cstride = (long long)d.ch * 3;   // one checkpoint column of histories
    const bool chan = tid < 2 * DK + DV;
    const int e = tid - (2 * DK + DV);
    int c = 0;
    if (tid < DK) c = kh * DK + tid;
    else if (tid < 2 * DK) c = d.hk * DK + kh * DK + (tid - DK);
    else if (chan) c = 2 * d.hk * DK + h * DV + (tid - 2 * DK);
    TA hx[3], xr[kMaxVerify];
    typename TapVec<TA>::type wv;
    TA ul = from_f32<TA>(0.f), bl = from_f32<TA>(0.f);
    float alog = 0.f, dtb = 0.f;
    if (chan) {
#pragma unroll
        for (int k = 0; k < 3; ++k) hx[k] = src[(long long)c * 3 + k];
        wv = load_taps(w, c);
#pragma unroll
        for (int jj = 0; jj < kMaxVerify; ++jj)
            if (jj < K) xr[jj] = __ldg((const TA *)a.x + (long long)(n * K + jj) * a.ld_x + c);
    } else {
#pragma unroll
        for (int jj = 0; jj < kMaxVerify; ++jj)
            if (jj < K) xr[jj] = __ldg((const TA *)a.z + (long long)(n * K + jj) * a.ld_z + (long long)h * DV + e);
        if (e < K) {
            ul = ((const TA *)a.u + (long long)(n * K + e) * a.ld_ub)[h];
            bl = ((const TA *)a.b_logit + (long long)(n * K + e) * a.ld_ub)[h];
            alog = a.A_log[h];
            dtb = a.dt_bias[h];
        }
    }
    // ---- conv + SiLU (q, k raw; v), SiLU(z), the gates: k records in shared memory
    if (chan) {
        float t[4];
        taps_f32(wv, t);
        float x0 = to_f32(hx[0]), x1 = to_f32(hx[1]), x2 = to_f32(hx[2]);
        const int off = tid < DK ? R.q + tid : (tid < 2 * DK ? R.k + (tid - DK) : R.v + (tid - 2 * DK));
#pragma unroll
        for (int jj = 0; jj < kMaxVerify; ++jj) {
            if (jj >= K) break;
            const float xc = to_f32(xr[jj]);
            const float acc = t[0] * x0 + t[1] * x1 + t[2] * x2 + t[3] * xc;
            x0 = x1;
            x1 = x2;
            x2 = xc;
            recs[jj * R.size + off] = silu_f(acc);
        }
    } else {
#pragma unroll
        for (int jj = 0; jj < kMaxVerify; ++jj)
            if (jj < K) recs[jj * R.size + R.z + e] = silu_f(to_f32(xr[jj]));
        if (e < K) {
            const float gg = -expf(alog) * softplus_f(to_f32(ul) + dtb);
            recs[e * R.size + R.ga] = expf(gg);
            recs[e * R.size + R.gb] = sigmoid_f(to_f32(bl));
        }
    }
    // ---- checkpoint histories: after token j the channel's last three raw inputs.  Every CTA
    // of the cluster has consumed its source-history loads above before it arrives here.
    cluster_sync_all();
    if (chan && (tid >= 2 * DK || gi == 0)) {
        TA x0 = hx[0], x1 = hx[1], x2 = hx[2];
#pragma unroll
        for (int jj = 0; jj < kMaxVerify; ++jj) {
            if (jj >= K) break;
            x0 = x1;
            x1 = x2;
            x2 = xr[jj];
            TA *hc = cols + jj * cstride + (long long)c * 3;
            hc[0] = x0;
            hc[1] = x1;
            hc[2] = x2;
        }
    }
    __syncthreads();   // records (raw q, k) complete
    // ---- q/k L2 factors (warp p: token p/2, q if p is even, k if odd), then k.q
    for (int p = warp; p < 2 * K; p += NW) {
        const float *vec = recs + (p >> 1) * R.size + ((p & 1) ? R.k : R.q);
        float ss = 0.f;
        for (int i = lane; i < DK; i += 32) ss += vec[i] * vec[i];
        ss = warp_sum(ss);
        if (lane == 0) nfac[p] = rsqrtf(ss + d.l2_eps) * ((p & 1) ? 1.f : d.q_scale);
    }
    __syncthreads();
    for (int j = warp; j < K; j += NW) {
        float *rc = recs + j * R.size;
        const float fq = nfac[2 * j], fk = nfac[2 * j + 1];
        float kq = 0.f;
        for (int i = lane; i < DK; i += 32) {
            const float qn = rc[R.q + i] * fq, kn = rc[R.k + i] * fk;
            rc[R.q + i] = qn;
            rc[R.k + i] = kn;
            kq += qn * kn;
        }
        kq = warp_sum(kq);
        if (lane == 0) rc[R.kq] = kq;
    }
    const float *rec0 = recs;
    const float nwt = tid < DV ? a.norm_w[tid] : 0.f;
    {
        __syncthreads();   // records complete
        for (int j = 0; j < K; ++j) {
            const float *rc = rec0 + j * R.size;
            float kr[RPT], qr[RPT];
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
            *reinterpret_cast<float4 *>(&red_p[rg][c4]) = pp;
            *reinterpret_cast<float4 *>(&red_s[rg][c4]) = ss;
            __syncthreads();   // (A)
            const float ga = rc[R.ga], gb = rc[R.gb];
            float ov = 0.f;
            if (tid < DV) {
                float p = 0.f, s2 = 0.f;
#pragma unroll
                for (int r = 0; r < RPP; ++r) {
                    p += red_p[r][tid];
                    s2 += red_s[r][tid];
                }
                const float uu = gb * (rc[R.v + tid] - ga * p);
                up[tid] = uu;
                ov = ga * s2 + uu * rc[R.kq];
            }
            __syncthreads();   // (B)
            {
                float *Mc = a.state + ((long long)(ck + j) * d.hv + h) * DK * DV;   // column j
                const float4 u4 = *reinterpret_cast<const float4 *>(&up[c4]);
#pragma unroll
                for (int x = 0; x < RPT; ++x) {
                    m[x].x = ga * m[x].x + kr[x] * u4.x;
                    m[x].y = ga * m[x].y + kr[x] * u4.y;
                    m[x].z = ga * m[x].z + kr[x] * u4.z;
                    m[x].w = ga * m[x].w + kr[x] * u4.w;
                    *reinterpret_cast<float4 *>(Mc + (long long)(rg + x * RPP) * DV + c4) = m[x];
                }
            }
            if (tid < DV) {   // gated RMSNorm of token j's o for this head
                const float sq = warp_sum(ov * ov);
                if (lane == 0) npart[warp] = sq;
                asm volatile("bar.sync 1, %0;" :: "r"(DV) : "memory");
                float tot = 0.f;
#pragma unroll
                for (int wi = 0; wi < DV / 32; ++wi) tot += npart[wi];
                const float rs = rsqrtf(tot / (float)DV + d.norm_eps);
                out[(long long)(n * K + j) * d.hv * DV + (long long)h * DV + tid] =
                    from_f32<TOut>(ov * rs * nwt * rc[R.z + tid]);
            }
        }
    }
}

template <int DK, int DV, typename TA, typename TOut>
cudaError_t launch_verify_t(const DecodeArgs &a, cudaStream_t s) {
    const int heads = a.n * a.d.hv;
    const DecRec R(DK, DV, 1);
    const size_t smem = (size_t)a.k_tokens * R.size * sizeof(float);
    auto kern = verify_kernel<DK, DV, TA, TOut>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(heads);
    lc.blockDim = dim3(4 * DV);
    lc.dynamicSmemBytes = smem;
    lc.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;   // the v-heads of one q/k head
    at[0].val.clusterDim.x = a.d.grp;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    lc.attrs = at;
    lc.numAttrs = 1;
    return cudaLaunchKernelEx(&lc, kern, a);
}

template <int DK, int DV>
cudaError_t launch_verify_d(const DecodeArgs &a, bool in_bf16, bool out_bf16, cudaStream_t s) {
    if (in_bf16)
        return out_bf16 ? launch_verify_t<DK, DV, __nv_bfloat16, __nv_bfloat16>(a, s)
                        : launch_verify_t<DK, DV, __nv_bfloat16, float>(a, s);
    return out_bf16 ? launch_verify_t<DK, DV, float, __nv_bfloat16>(a, s)
                    : launch_verify_t<DK, DV, float, float>(a, s);
}

}  // namespace

cudaError_t launch_verify(const DecodeArgs &a, bool in_bf16, bool out_bf16, cudaStream_t s) {
    if (a.n == 0) return cudaSuccess;
    if (a.k_tokens < 1 || a.k_tokens > kMaxVerify || a.d.grp > 4 || !a.ckpt_idx)
        return cudaErrorInvalidValue;
    switch (a.d.dk) {
        case 32: return launch_verify_d<32, 32>(a, in_bf16, out_bf16, s);
        case 64: return launch_verify_d<64, 64>(a, in_bf16, out_bf16, s);
        case 128: return launch_verify_d<128, 128>(a, in_bf16, out_bf16, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
