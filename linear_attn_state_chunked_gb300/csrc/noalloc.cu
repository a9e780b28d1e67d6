// noalloc.cu -- hypic_segment_build_noalloc: the segment build for callers
// that are not allowed to allocate device memory.
//
// Some callers only ever receive input and output buffers: a plugin running
// inside a host inference engine that owns all device memory through its own
// pool and gives its kernels no allocator, or a latency-critical path where a
// cudaMalloc (which may synchronise the device) is not permitted.  They cannot
// provide the small workspace hypic_segment_build asks for, so this entry
// point uses a fixed scratch block compiled into the library instead.
//
// The scratch lives in this file as a static __device__ array: every GPU that
// loads the library holds it until the process exits.  Host code must not
// hand the array's name to a kernel (on the host it is only a stand-in, not a
// device address); the device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, on the first call made on
// that device.  All calls share the one block, so calls whose work overlaps
// on the GPU race on it.
#include <cstdio>
#include <mutex>

#include "kernels.h"

namespace hypic {
int report_error(int code, const char *msg);  // api.cu: sets hypic_last_error()
}

namespace {

// Maximum scratch this entry point can serve: one build workspace.
constexpr size_t kScratchBytes = 256;
static __device__ __align__(256) unsigned char g_build_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::once_flag g_once[kMaxDevices];
void *g_scratch_ptr[kMaxDevices];
cudaError_t g_scratch_err[kMaxDevices];

}  // namespace

namespace {

// This device's scratch address, looked up on first use (see above).
int scratch_of_current_device(void **out)
{
    char msg[256];
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        snprintf(msg, sizeof(msg), "cudaGetDevice: %s", cudaGetErrorString(e));
        return hypic::report_error(HYPIC_ERR_CUDA, msg);
    }
    if (dev < 0 || dev >= kMaxDevices) {
        snprintf(msg, sizeof(msg), "device %d beyond the %d devices this entry point serves", dev, kMaxDevices);
        return hypic::report_error(HYPIC_ERR_UNSUPPORTED, msg);
    }
    std::call_once(g_once[dev], [dev]() {
        void *p = nullptr;
        g_scratch_err[dev] = cudaGetSymbolAddress(&p, g_build_scratch);
        g_scratch_ptr[dev] = p;
    });
    if (g_scratch_err[dev] != cudaSuccess || !g_scratch_ptr[dev]) {
        snprintf(msg, sizeof(msg), "cudaGetSymbolAddress of the static scratch on device %d: %s", dev,
                 cudaGetErrorString(g_scratch_err[dev]));
        return hypic::report_error(HYPIC_ERR_CUDA, msg);
    }
    *out = g_scratch_ptr[dev];
    return HYPIC_OK;
}

}  // namespace

extern "C" int hypic_noalloc_status(hypic_stream stream)
{
    void *scratch = nullptr;
    const int rc = scratch_of_current_device(&scratch);
    if (rc != HYPIC_OK) return rc;
    // the scratch is laid out like a build workspace: its status word is the
    // one hypic_workspace_status reads
    return hypic_workspace_status(scratch, stream);
}

extern "C" int hypic_segment_build_noalloc(const hypic_desc *desc, const hypic_tokens *tok,
                                           const int64_t *seg_off, int32_t n_seg, float *T_out,
                                           float *S_out, hypic_stream stream)
{
    char msg[256];
    const size_t need = hypic_workspace_size(desc);
    if (need > kScratchBytes) {
        snprintf(msg, sizeof(msg),
                 "this build needs %zu bytes of scratch; the library's static scratch holds %zu",
                 need, kScratchBytes);
        return hypic::report_error(HYPIC_ERR_WORKSPACE, msg);
    }
    void *scratch = nullptr;
    const int rc = scratch_of_current_device(&scratch);
    if (rc != HYPIC_OK) return rc;
    // The build clears what must start at zero (its status word) on `stream`
    // before its kernel runs.
    return hypic_segment_build(desc, tok, seg_off, n_seg, T_out, S_out, scratch, kScratchBytes, stream);
}
