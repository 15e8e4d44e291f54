// gdn_verify.cu -- multi-token verification decode (hyperflare core-design,
// speculative target state: eight recurrent checkpoint columns per request, a
// round writes the columns of its verification inputs, and the committed
// column is the one of the last accepted input).
//
// For sequence n with k tokens t_0 .. t_{k-1} and source slot s, the
// one-token rule of gdn_decode.cu is applied k times in a row, starting from
// state and conv history of slot s (read only); after token j the state and
// the conv history (its last three raw inputs) are written to slot
// ckpt_idx[n] + j, and y_j is the gated-norm output of token j.  Two
// launches, like the fused decode:
//  - verify_prep_kernel, one CTA per (sequence, q/k head) unit: the conv
//    over the k tokens from the source history (writing every column's
//    history), SiLU, the q/k L2 norms, k.q, the gates and SiLU(z), as one
//    record per (unit, token) in the caller's workspace;
//  - verify_kernel, one CTA per (sequence, v-head): the unit's k records are
//    staged in shared memory, the head state is read once into registers
//    (thread: one float4 column group of RPT rows) and carried through the k
//    tokens; every token's state goes straight from registers to its column.
//    HBM bytes per head: (1 + k) * dk*dv*4.
#include "gdn_common.cuh"

namespace gdn {

namespace {

template <int DK, int DV, typename TA>
__global__ void __launch_bounds__(256) verify_prep_kernel(DecodeArgs a) {
    __shared__ __align__(16) float qs[kMaxVerify][DK], ks[kMaxVerify][DK];
    const Dims &d = a.d;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // verify_kernel may be scheduled once every prep CTA has started: it loads its head
    // state first and waits for this grid's completion before it reads a record
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int u = blockIdx.x, n = u / d.hk, kh = u % d.hk, G = d.grp, K = a.k_tokens;
    const DecRec R(DK, DV, G);
    float *rec0 = a.ws + (long long)u * K * R.size;
    const int slot = slot_of(a.state_idx, n, d.n_slots, a.err);
    int ck = -1;
    if (slot >= 0) {
        ck = a.ckpt_idx[n];
        if (ck < 0 || ck + K > d.n_slots) {
            if (tid == 0) set_error(a.err, GDN_DEVERR_SLOT);
            ck = -1;
        }
    }
    if (slot < 0 || ck < 0) {   // padding lane, or checkpoint columns out of range
        if (tid < K) rec0[tid * R.size + R.slot] = __int_as_float(-1);
        return;
    }
    const TA *w = (const TA *)a.conv_w;
    const TA *src = (const TA *)a.conv_state + (long long)slot * d.ch * 3;
    TA *cols = (TA *)a.conv_state + (long long)ck * d.ch * 3;
    const long long cstride = (long long)d.ch * 3;   // one checkpoint column of histories
    const int nch = 2 * DK + G * DV;
    for (int ci = tid; ci < nch; ci += 256) {
        int c;
        if (ci < DK) c = kh * DK + ci;
        else if (ci < 2 * DK) c = d.hk * DK + kh * DK + (ci - DK);
        else c = 2 * d.hk * DK + kh * G * DV + (ci - 2 * DK);
        const float w0 = to_f32(w[c * 4 + 0]), w1 = to_f32(w[c * 4 + 1]), w2 = to_f32(w[c * 4 + 2]),
                    w3 = to_f32(w[c * 4 + 3]);
        TA x0 = src[(long long)c * 3], x1 = src[(long long)c * 3 + 1], x2 = src[(long long)c * 3 + 2];
        TA xr[kMaxVerify];   // the k raw inputs of this channel, loads issued together
#pragma unroll
        for (int j = 0; j < kMaxVerify; ++j)
            if (j < K) xr[j] = __ldg((const TA *)a.x + (long long)(n * K + j) * a.ld_x + c);
#pragma unroll
        for (int j = 0; j < kMaxVerify; ++j) {
            if (j >= K) break;
            const TA xc = xr[j];
            const float acc = w0 * to_f32(x0) + w1 * to_f32(x1) + w2 * to_f32(x2) + w3 * to_f32(xc);
            x0 = x1;
            x1 = x2;
            x2 = xc;
            TA *hc = cols + j * cstride + (long long)c * 3;   // history after token j
            hc[0] = x0;
            hc[1] = x1;
            hc[2] = x2;
            const float val = silu_f(acc);
            if (ci < DK) qs[j][ci] = val;
            else if (ci < 2 * DK) ks[j][ci - DK] = val;
            else rec0[j * R.size + R.v + (ci - 2 * DK)] = val;
        }
    }
    {   // SiLU(z) of the unit's v-heads for the k tokens: every load issued before any store
        constexpr int ZMAX = kMaxVerify * 4 * DV / 256;   // k <= 8, G <= 4
        TA zr[ZMAX];
#pragma unroll
        for (int i = 0; i < ZMAX; ++i) {
            const int e = tid + 256 * i;
            if (e < K * G * DV) {
                const int j = e / (G * DV), idx = e % (G * DV);
                zr[i] = __ldg((const TA *)a.z + (long long)(n * K + j) * a.ld_z + (long long)kh * G * DV + idx);
            }
        }
#pragma unroll
        for (int i = 0; i < ZMAX; ++i) {
            const int e = tid + 256 * i;
            if (e < K * G * DV) {
                const int j = e / (G * DV), idx = e % (G * DV);
                rec0[j * R.size + R.z + idx] = silu_f(to_f32(zr[i]));
            }
        }
    }
    if (tid < K * G) {
        const int j = tid / G, gi = tid % G, h = kh * G + gi;
        const TA *uv = (const TA *)a.u + (long long)(n * K + j) * a.ld_ub;
        const TA *bv = (const TA *)a.b_logit + (long long)(n * K + j) * a.ld_ub;
        const float gg = -expf(a.A_log[h]) * softplus_f(to_f32(uv[h]) + a.dt_bias[h]);
        rec0[j * R.size + R.ga + gi] = expf(gg);
        rec0[j * R.size + R.gb + gi] = sigmoid_f(to_f32(bv[h]));
    }
    __syncthreads();
    // warp j: the L2 norms of token j's q and k, then q, k and k.q into its record
    for (int j = warp; j < K; j += 8) {
        float sq = 0.f, sk = 0.f;
        for (int i = lane; i < DK; i += 32) {
            sq += qs[j][i] * qs[j][i];
            sk += ks[j][i] * ks[j][i];
        }
        sq = warp_sum(sq);
        sk = warp_sum(sk);
        const float fq = rsqrtf(sq + d.l2_eps) * d.q_scale, fk = rsqrtf(sk + d.l2_eps);
        float *rc = rec0 + j * R.size;
        float kq = 0.f;
        for (int i = lane; i < DK; i += 32) {
            const float qn = qs[j][i] * fq, kn = ks[j][i] * fk;
            rc[R.q + i] = qn;
            rc[R.k + i] = kn;
            kq += qn * kn;
        }
        kq = warp_sum(kq);
        if (lane == 0) {
            rc[R.kq] = kq;
            rc[R.slot] = __int_as_float(slot);
        }
    }
}

template <int DK, int DV, typename TOut>
__global__ void __launch_bounds__(4 * DV, 2) verify_kernel(DecodeArgs a) {
    constexpr int NT = 4 * DV, LPR = DV / 4, RPP = NT / LPR, RPT = DK / RPP;
    extern __shared__ __align__(16) float recs[];   // the unit's k records
    __shared__ __align__(16) float red_p[RPP][DV];
    __shared__ __align__(16) float red_s[RPP][DV];
    __shared__ __align__(16) float up[DV];
    __shared__ float npart[DV / 32];
    const Dims &d = a.d;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // one CTA per (sequence, v-head); its q/k head's unit holds the records
    const int G = d.grp, K = a.k_tokens;
    const int n = blockIdx.x / d.hv, h = blockIdx.x % d.hv, kh = h / G, gi = h % G;
    const int u = n * d.hk + kh;
    const DecRec R(DK, DV, G);
    const float *grec = a.ws + (long long)u * K * R.size;
    TOut *out = (TOut *)a.out;
    // the head state does not depend on the prep grid: its loads go out first
    const int rg = tid / LPR, c4 = (tid % LPR) * 4;
    const int sslot = slot_of(a.state_idx, n, d.n_slots, nullptr);
    float4 m[RPT];
    if (sslot >= 0) {
        const float *Ms = a.state + ((long long)sslot * d.hv + h) * DK * DV;
#pragma unroll
        for (int x = 0; x < RPT; ++x)
            m[x] = *reinterpret_cast<const float4 *>(Ms + (long long)(rg + x * RPP) * DV + c4);
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int slot = __float_as_int(grec[R.slot]);
    if (slot < 0) {   // padding lane (or rejected columns): zero outputs, no state traffic
        for (int e = tid; e < K * DV; e += NT) {
            const int j = e / DV, idx = e % DV;
            out[(long long)(n * K + j) * d.hv * DV + (long long)h * DV + idx] = from_f32<TOut>(0.f);
        }
        return;
    }
    const int ck = a.ckpt_idx[n];
    // every record of the unit into shared memory at once (R.size is a multiple of 4 floats)
    for (int e4 = tid; e4 < K * R.size / 4; e4 += NT)
        reinterpret_cast<float4 *>(recs)[e4] = reinterpret_cast<const float4 *>(grec)[e4];
    const float *rec0 = recs;
    const float nwt = tid < DV ? a.norm_w[tid] : 0.f;
    {
        __syncthreads();   // records staged
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
            const float ga = rc[R.ga + gi], gb = rc[R.gb + gi];
            float ov = 0.f;
            if (tid < DV) {
                float p = 0.f, s2 = 0.f;
#pragma unroll
                for (int r = 0; r < RPP; ++r) {
                    p += red_p[r][tid];
                    s2 += red_s[r][tid];
                }
                const float uu = gb * (rc[R.v + gi * DV + tid] - ga * p);
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
                    from_f32<TOut>(ov * rs * nwt * rc[R.z + gi * DV + tid]);
            }
        }
    }
}

template <int DK, int DV, typename TA, typename TOut>
cudaError_t launch_verify_t(const DecodeArgs &a, cudaStream_t s) {
    const int units = a.n * a.d.hk;
    verify_prep_kernel<DK, DV, TA><<<units, 256, 0, s>>>(a);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int heads = a.n * a.d.hv;
    const DecRec R(DK, DV, a.d.grp);
    const size_t smem = (size_t)a.k_tokens * R.size * sizeof(float);
    auto kern = verify_kernel<DK, DV, TOut>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t lc = {};
    lc.gridDim = dim3(heads);
    lc.blockDim = dim3(4 * DV);
    lc.dynamicSmemBytes = smem;
    lc.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // overlap the prep's tail
    at[0].val.programmaticStreamSerializationAllowed = 1;
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

size_t verify_ws_bytes(const Dims &d, long long tokens) {
    const DecRec R(d.dk, d.dv, d.grp);
    return (size_t)(tokens > 0 ? tokens : 0) * d.hk * R.size * sizeof(float);
}

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
