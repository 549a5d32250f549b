// build_noalloc.cu -- hypic_segment_build_noalloc: the segment build for
// callers that may not allocate device memory.  Its scratch (the longest-
// body-first work order and the work counter) lives in a fixed array owned
// by this library on every device that loads it, instead of in a caller
// workspace.  Everything else is hypic_segment_build itself.
#include <cuda_runtime.h>
#include <stdio.h>

#include "../../include/hypic.h"
#include "kernels.h"

namespace hypic {
void set_detail(const char* msg);  // api.cu: sets hypic_last_error_detail()
hypic_status segment_build_impl(const hypic_build_args* args, void* workspace, size_t workspace_bytes,
                                hypic_stream_t stream, bool tables);  // api.cu
}

namespace {

// Same layout as the caller workspace of hypic_segment_build: the order
// (int32 per segment, padded to 256 bytes) then a 256-byte counter block.
constexpr size_t kNoallocBytes = ((size_t)HYPIC_NOALLOC_MAX_SEGMENTS * 4 + 255) / 256 * 256 + 256;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocBytes];

// Device address of g_noalloc_scratch on the current device (the host-side
// symbol is only a stand-in for it), looked up on every call with that device
// current: a cheap host-side query, and never stale after a device reset.
void* scratch_address(cudaError_t* err) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    return *err == cudaSuccess ? p : nullptr;
}

}  // namespace

extern "C" hypic_status hypic_segment_build_noalloc(const hypic_build_args* args, hypic_stream_t stream) {
    char msg[256];
    if (args && args->n_segments > HYPIC_NOALLOC_MAX_SEGMENTS) {
        snprintf(msg, sizeof(msg),
                 "no-alloc build: %d segments exceed the fixed scratch limit of %d (use hypic_segment_build "
                 "with a caller workspace)",
                 args->n_segments, HYPIC_NOALLOC_MAX_SEGMENTS);
        hypic::set_detail(msg);
        return HYPIC_ERR_WORKSPACE;
    }
    if (hypic_build_workspace_size(args) == 0) return hypic_segment_build(args, nullptr, 0, stream);  // the argument error
    // The plan and counter only: KDA, whose tensor-core path needs its chunk tables, runs its CUDA-core
    // kernel here.
    const size_t need = hypic::build_workspace_bytes(args->n_segments);
    if (need > kNoallocBytes) {
        snprintf(msg, sizeof(msg), "no-alloc build: needs %zu bytes of scratch, the fixed array holds %zu", need,
                 kNoallocBytes);
        hypic::set_detail(msg);
        return HYPIC_ERR_WORKSPACE;
    }
    cudaError_t e;
    void* ws = scratch_address(&e);
    if (!ws) {
        snprintf(msg, sizeof(msg), "no-alloc build: address of the fixed scratch: %s", cudaGetErrorString(e));
        hypic::set_detail(msg);
        return HYPIC_ERR_CUDA;
    }
    return hypic::segment_build_impl(args, ws, kNoallocBytes, stream, false);
}
