// gdn_state.cu -- slot maintenance: snapshot, restore, initialise and reset
// of recurrent states and conv histories as one indirect copy driven by
// device-resident slot indices (hyperflare core-design: "State operations" of
// the native model contract; the speculative-state section's snapshot of one
// state column together with its three-token conv window).  A pure HBM
// stream: every 16-byte word of a moved slot is read once and written once.
#include "gdn_common.cuh"

namespace gdn {
namespace {

constexpr int SC_NT = 256;     // threads per block
constexpr int SC_U = 4;        // 16-byte words in flight per thread

// Block (x, i) moves its share of pair i: words x*NT + tid + k*gridDim.x*NT of
// the destination slot's state, then of its history (loads of one round all
// issued before the stores).  A reset writes zeros and reads nothing.
__global__ void __launch_bounds__(SC_NT) state_copy_kernel(
    const uint4 *src_state, uint4 *dst_state, long long state_words, const uint4 *src_conv,
    uint4 *dst_conv, long long conv_words, int n_src, int n_dst, const int32_t *src_idx,
    const int32_t *dst_idx, unsigned *err) {
    const int i = blockIdx.y;
    const int t = dst_idx[i];
    if (t < 0) return;                                   // inactive lane
    const int s = src_idx[i];
    if (t >= n_dst || (s >= n_src && (src_state || src_conv))) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_error(err, GDN_DEVERR_SLOT);
        return;
    }
    auto move = [&](const uint4 *src, uint4 *dst, long long words) {
        if (!dst) return;
        uint4 *dp = dst + (long long)t * words;
        const uint4 *sp = (s >= 0 && src) ? src + (long long)s * words : nullptr;
        const long long stride = (long long)gridDim.x * SC_NT;
        for (long long w0 = (long long)blockIdx.x * SC_NT + threadIdx.x; w0 < words; w0 += stride * SC_U) {
            uint4 v[SC_U];
#pragma unroll
            for (int u = 0; u < SC_U; ++u) {
                const long long w = w0 + u * stride;
                v[u] = make_uint4(0u, 0u, 0u, 0u);
                if (sp && w < words) v[u] = __ldcs(sp + w);
            }
#pragma unroll
            for (int u = 0; u < SC_U; ++u) {
                const long long w = w0 + u * stride;
                if (w < words) __stcs(dp + w, v[u]);
            }
        }
    };
    move(src_state, dst_state, state_words);
    move(src_conv, dst_conv, conv_words);
}

}  // namespace

cudaError_t launch_state_copy(const Dims &d, bool act_bf16, const float *src_state,
                              const void *src_conv, int n_src, float *dst_state, void *dst_conv,
                              int n_dst, const int32_t *src_idx, const int32_t *dst_idx, int n,
                              unsigned *err, cudaStream_t s) {
    if (n <= 0 || (!dst_state && !dst_conv)) return cudaSuccess;
    const long long sw = (long long)d.hv * d.dk * d.dv * 4 / 16;               // words per state slot
    const long long cw = (long long)d.ch * 3 * (act_bf16 ? 2 : 4) / 16;         // per history slot
    const long long most = dst_state ? (dst_conv && cw > sw ? cw : sw) : cw;
    long long gx = (most + (long long)SC_NT * SC_U - 1) / ((long long)SC_NT * SC_U);
    if (gx < 1) gx = 1;
    if (gx > 1024) gx = 1024;
    state_copy_kernel<<<dim3((unsigned)gx, (unsigned)n), SC_NT, 0, s>>>(
        (const uint4 *)src_state, (uint4 *)dst_state, sw, (const uint4 *)src_conv,
        (uint4 *)dst_conv, cw, n_src, n_dst, src_idx, dst_idx, err);
    return cudaGetLastError();
}

}  // namespace gdn
