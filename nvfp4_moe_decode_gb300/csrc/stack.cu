// stack.cu -- the residual add that closes a pre-norm decoder stack of MoE
// layers (the last layer's output added to the residual stream).
//
// Flint page ("vLLM adds day-0 support for Recursive's Flint"), section
// "A 40B MoE that activates 2.5B parameters": a 47-layer pre-norm decoder.
// Each layer's own residual add and RMSNorm run in the prologue of the next
// layer kernel (layer.cu); only the final add needs a kernel of its own.
#include "kernels.cuh"

namespace moe {

// out = bf16(a + b), elementwise over n bf16 values (n % 8 == 0).
__global__ void residual_add_kernel(const __nv_bfloat16 *a, const __nv_bfloat16 *b, __nv_bfloat16 *out, int n)
{
    griddep_wait();
    const int n8 = n / 8;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += gridDim.x * blockDim.x) {
        uint4 x = reinterpret_cast<const uint4 *>(a)[i];
        const uint4 y = reinterpret_cast<const uint4 *>(b)[i];
        uint32_t *xw = &x.x;
        const uint32_t *yw = &y.x;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const __nv_bfloat16 lo = __float2bfloat16_rn(bf16_bits_to_float(xw[q] & 0xFFFFu) + bf16_bits_to_float(yw[q] & 0xFFFFu));
            const __nv_bfloat16 hi = __float2bfloat16_rn(bf16_bits_to_float(xw[q] >> 16) + bf16_bits_to_float(yw[q] >> 16));
            xw[q] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
        }
        reinterpret_cast<uint4 *>(out)[i] = x;
    }
    griddep_launch();
}

cudaError_t launch_residual_add(const __nv_bfloat16 *a, const __nv_bfloat16 *b, __nv_bfloat16 *out, int n,
                                cudaStream_t stream, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    const int n8 = n / 8;
    cfg.gridDim = dim3((n8 + 255) / 256 > 0 ? (n8 + 255) / 256 : 1);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, residual_add_kernel, a, b, out, n);
}

}  // namespace moe
