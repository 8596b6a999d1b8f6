// conv_fwd_noalloc.cu -- conv_fwd for callers that must not allocate device
// memory: the scratch conv_fwd needs comes from a fixed array compiled into
// this library instead of from a caller-provided workspace.  That scratch has
// up to three regions, laid out as conv_fwd lays out its workspace: the
// filters re-laid as pre-split tensor-core tiles (the B image); for the patch
// and space-to-depth forms, the channel-blocked or space-to-depth copy of x,
// whose size grows with the batch; and the partial tiles of a split last
// round of tiles.  Shapes whose total exceeds the array are refused.
//
// Who needs this: code that runs under a device-memory manager owning the
// whole heap (a host framework, an embedded runtime with a fixed budget), or
// a latency-critical loop where an allocation's implicit device
// synchronisation is not acceptable.  Such a caller can pass inputs and
// outputs it already owns, but cannot obtain a workspace.
//
// The array is a file-scope __device__ variable: every device that loads the
// library holds one copy of it until the process exits.  Host code cannot use
// the array's name as a device address (it names a host-side shadow), so the
// first call on each device looks up the real address with
// cudaGetSymbolAddress, with that device current, and caches it.
#include <mutex>

#include "conv_b200_internal.h"

namespace cb200 {
namespace {

__device__ __align__(256) unsigned char g_fwd_scratch[CONV_FWD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices];
cudaError_t g_scratch_err[kMaxDevices];
std::once_flag g_scratch_once[kMaxDevices];

void resolve_scratch(int dev)
{
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_fwd_scratch);
    g_scratch_err[dev] = e;
    g_scratch_addr[dev] = (e == cudaSuccess) ? p : nullptr;
    if (e != cudaSuccess) cudaGetLastError();
}

}  // namespace
}  // namespace cb200

extern "C" int conv_fwd_noalloc(const conv_shape_t* s, const float* x, const float* w, const float* b, float* y,
                                conv_stream_t stream)
{
    using namespace cb200;
    // Shapes whose scratch (B image + staged copy of x + split partials) does
    // not fit are refused before anything is launched.  (An invalid shape
    // needs 0 bytes here and is reported by conv_fwd's own validation below.)
    const size_t need = conv_b200_workspace_bytes(CONV_OP_FWD, s);
    if (need > size_t(CONV_FWD_NOALLOC_SCRATCH_BYTES)) return CONV_ERR_SCRATCH_LIMIT;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return CONV_ERR_DEVICE;
    }
    std::call_once(g_scratch_once[dev], resolve_scratch, dev);
    if (g_scratch_err[dev] != cudaSuccess || g_scratch_addr[dev] == nullptr) return CONV_ERR_CUDA;
    // Every region is written in full by this call before it is read: the B
    // image (padding included) by its builder, the copy of x by its gather
    // kernel, and each partial tile by the GEMM piece that owns it before the
    // reduce adds them.  So nothing an earlier call left in the array needs
    // clearing.
    return conv_fwd(s, x, w, b, y, g_scratch_addr[dev], size_t(CONV_FWD_NOALLOC_SCRATCH_BYTES), stream);
}
