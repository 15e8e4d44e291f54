// gdn_noalloc.cu -- gdn_mixer_prefill_static: the fused prefill for callers
// that cannot allocate device memory.
//
// gdn_mixer_prefill needs a caller-provided workspace for its intermediates
// (the fp32 conv output, the gates and the fp32 mixer output before the norm).
// Some callers have no way to provide one: code that runs where every device
// allocation is forbidden after start-up (a serving step loop, an allocation-
// free plugin that is handed only a stream and its tensors), or a host runtime
// without a device allocator of its own.  This entry point takes the same
// arguments minus the workspace and keeps the intermediates in a fixed array
// compiled into the library instead.  It allocates nothing and calls no
// allocating routine.
//
// The array is file-scope device memory of GDN_STATIC_SCRATCH_BYTES; every
// GPU that loads the library holds it until the process exits.  Host code
// cannot use the array's name as a device address, so the address is looked
// up once per device with cudaGetSymbolAddress (on the first call made while
// that device is current) and cached; make that first call before any stream
// capture.  The cache lives as long as the device's context: after
// cudaDeviceReset (or any teardown of the primary context) the cached address
// is stale, so a process that resets a device must not call this entry point
// on it again.  All calls share the one array and it keeps the last call's
// contents: two calls whose work overlaps on the GPU (different streams, or
// different host threads) race on it and must be serialised by the caller.
// Nothing in it needs to start at zero: every intermediate a call reads is
// written earlier in the same call.
#include <mutex>

#include "gdn_common.cuh"

namespace {

constexpr size_t kScratchBytes = GDN_STATIC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_prefill_scratch[kScratchBytes];

constexpr int kMaxDev = 64;
void *g_scratch_addr[kMaxDev];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (set up once per device).
gdn_status scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return GDN_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress((void **)&ptr, g_prefill_scratch) != cudaSuccess || !ptr)
            return GDN_ERR_CUDA;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_mixer_prefill_static(const gdn_config *cfg, const gdn_mixer_io *io,
                                               void *stream) {
    if (!cfg || !io || io->T < 0 || io->n_seqs < 0) return GDN_ERR_INVALID_ARG;
    if (gdn_workspace_size(cfg, io->T, io->n_seqs) == 0)
        return gdn_mixer_prefill(cfg, io, nullptr, 0, stream);  // the configuration's own status
    // only the prefill's own intermediates have to fit
    if (gdn::mixer_prefill_ws_bytes(cfg, io->T, io->n_seqs) > kScratchBytes)
        return GDN_ERR_WORKSPACE;   // too many tokens for the fixed scratch
    void *ws = nullptr;
    const gdn_status st = scratch_address(&ws);
    if (st != GDN_OK) return st;
    return gdn_mixer_prefill(cfg, io, ws, kScratchBytes, stream);
}
