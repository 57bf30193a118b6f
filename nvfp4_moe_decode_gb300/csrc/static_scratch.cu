// static_scratch.cu -- moe_layer_forward_static: the layer with its scratch in
// a fixed device array inside the library, for callers that cannot allocate.
//
// Some callers can hand the layer only its inputs and outputs: a plugin or
// custom-op interface whose signature carries no workspace, or a process that
// fixes its device-memory budget at start-up and forbids allocation on the
// serving path.  They cannot own the workspace that moe_layer_forward takes,
// so this entry point uses a file-scope __device__ array instead.  It
// allocates nothing: no cudaMalloc/cudaFree, no allocating library routine.
// The array is part of the module image, loaded with the library.
//
// The scratch is one per device (per context), so calls on one device must
// not overlap: two calls in flight at once (two streams, two host threads)
// share the counters and buffers and race.  Serialise them on one stream or
// with events.
//
// The caller cannot zero this scratch, so a call that gave up on a bounded
// wait must not leave it unusable: every call first enqueues the library's
// re-arm kernel, which clears the counters and advances the launch tag when
// the scratch's flag word reports a timeout (and does nothing otherwise).
// moe_static_read_device_flag reads and clears that flag word.
#include <mutex>

#include "kernels.cuh"

using namespace moe;

namespace {

// Sized for the largest decode batch (MOE_MAX_DECODE_T tokens): routing
// results, SiLU*up activations, per-expert partials and the control words.
constexpr size_t STATIC_SCRATCH_BYTES = MOE_STATIC_SCRATCH_BYTES;

static __device__ __align__(256) uint8_t g_scratch[STATIC_SCRATCH_BYTES];

constexpr int MAX_DEVICES = 64;
std::mutex g_setup_mutex;
void *g_scratch_ptr[MAX_DEVICES] = {nullptr};

// First call on a device: look up the array's address with that device
// current, and zero it on the caller's stream (the control words must start
// at zero; static device memory already does, this makes it explicit).
moe_status scratch_for_current_device(cudaStream_t stream, void **ptr)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (dev < 0 || dev >= MAX_DEVICES)
        return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr)
            return MOE_ERR_CUDA;
        if (cudaMemsetAsync(p, 0, STATIC_SCRATCH_BYTES, stream) != cudaSuccess)
            return MOE_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return MOE_OK;
}

}  // namespace

extern "C" moe_status moe_static_read_device_flag(moe_stream_t stream, uint32_t *flag_out)
{
    if (!flag_out)
        return MOE_ERR_INVALID_ARG;
    void *scratch = nullptr;
    const moe_status s = scratch_for_current_device((cudaStream_t)stream, &scratch);
    if (s != MOE_OK)
        return s;
    return moe_read_device_flag(scratch, stream, flag_out);
}

extern "C" moe_status moe_layer_forward_static(const void *x, const void *router_w,
                                               const moe_expert_bank *routed,
                                               const moe_expert_bank *shared, void *out, int T,
                                               moe_stream_t stream)
{
    // the scratch covers T <= MOE_MAX_DECODE_T only
    if (T < 1 || T > MOE_MAX_DECODE_T)
        return MOE_ERR_UNSUPPORTED;
    const size_t need = moe_workspace_bytes(T);
    if (need > STATIC_SCRATCH_BYTES)
        return MOE_ERR_WORKSPACE;
    void *scratch = nullptr;
    moe_status s = scratch_for_current_device((cudaStream_t)stream, &scratch);
    if (s != MOE_OK)
        return s;
    // the re-arm kernel first: recovery from an earlier call's wait timeout
    return layer_forward(x, router_w, routed, shared, out, T, scratch, STATIC_SCRATCH_BYTES, (cudaStream_t)stream,
                         true);
}
