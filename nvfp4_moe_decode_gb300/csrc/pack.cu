// pack.cu -- load-time repacking of NVFP4 matrices (canonical -> packed and
// back) and a dequantiser that reads the packed form through the same
// in-register decode as the GEMV kernels.
//
// Flint page ("vLLM adds day-0 support for Recursive's Flint"), section
// "A 40B MoE that activates 2.5B parameters": the checkpoint's NVFP4 blocks
// are repacked losslessly at load time.  Section "From 1,096 kernels to 346":
// one packed NVFP4 layout serves the small-batch GEMVs.  The layout itself is
// documented in common.cuh.
#include "kernels.cuh"

namespace moe {


// One thread per packed byte: gather its two nibbles (or its scale byte).
__global__ void pack_kernel(PackArgs a)
{
    const size_t per_mat = (size_t)a.N * a.K * 9 / 16;
    const size_t total = per_mat * a.count;
    const size_t bb = band_bytes(a.K);
    for (size_t o = (size_t)blockIdx.x * blockDim.x + threadIdx.x; o < total;
         o += (size_t)gridDim.x * blockDim.x) {
        const size_t m = o / per_mat, r = o % per_mat;
        const int b = (int)(r / bb), off = (int)(r % bb);
        const uint8_t *codes = a.codes + m * (size_t)a.N * (a.K / 2);
        const uint8_t *scales = a.scales + m * (size_t)a.N * (a.K / 16);
        uint8_t v;
        if (!is_scale_byte(off)) {
            v = 0;
            for (int nib = 0; nib < 2; ++nib) {
                int i, k;
                code_element(off, nib, i, k);
                const int n = band_row_to_matrix_row(a.kind, a.N, b, i);
                const uint8_t cb = codes[(size_t)n * (a.K / 2) + k / 2];
                const uint8_t code = (k & 1) ? (cb >> 4) : (cb & 15);
                v |= (uint8_t)(code << (4 * nib));
            }
        } else {
            int i, bk;
            scale_element(off, i, bk);
            const int n = band_row_to_matrix_row(a.kind, a.N, b, i);
            v = scales[(size_t)n * (a.K / 16) + bk];
        }
        a.packed[o] = v;
    }
}


// One thread per canonical code byte, then one per scale byte.
__global__ void unpack_kernel(UnpackArgs a)
{
    const size_t code_per = (size_t)a.N * (a.K / 2), scale_per = (size_t)a.N * (a.K / 16);
    const size_t per_mat = (size_t)a.N * a.K * 9 / 16;
    const size_t bb = band_bytes(a.K);
    const size_t total = (code_per + scale_per) * a.count;
    for (size_t o = (size_t)blockIdx.x * blockDim.x + threadIdx.x; o < total;
         o += (size_t)gridDim.x * blockDim.x) {
        if (o < code_per * a.count) {
            const size_t m = o / code_per, r = o % code_per;
            const int n = (int)(r / (a.K / 2)), jb = (int)(r % (a.K / 2));
            int b, i;
            matrix_row_to_band(a.kind, a.N, n, b, i);
            uint8_t v = 0;
            for (int h = 0; h < 2; ++h) {
                int off, nib;
                code_position(i, 2 * jb + h, off, nib);
                const uint8_t pb = a.packed[m * per_mat + (size_t)b * bb + off];
                const uint8_t code = nib ? (pb >> 4) : (pb & 15);
                v |= (uint8_t)(code << (4 * h));
            }
            a.codes[o] = v;
        } else {
            const size_t o2 = o - code_per * a.count;
            const size_t m = o2 / scale_per, r = o2 % scale_per;
            const int n = (int)(r / (a.K / 16)), bk = (int)(r % (a.K / 16));
            int b, i;
            matrix_row_to_band(a.kind, a.N, n, b, i);
            a.scales[o2] = a.packed[m * per_mat + (size_t)b * bb + scale_position(i, bk)];
        }
    }
}


// out[n][k] = e2m1 * e4m3 * tscale, decoding the code byte exactly as the
// GEMV kernels do (cvt.rn.f16x2.e2m1x2 on the byte that holds the element).
__global__ void dequant_kernel(DequantArgs a)
{
    const size_t total = (size_t)a.N * a.K;
    const size_t bb = band_bytes(a.K);
    for (size_t o = (size_t)blockIdx.x * blockDim.x + threadIdx.x; o < total;
         o += (size_t)gridDim.x * blockDim.x) {
        const int n = (int)(o / a.K), k = (int)(o % a.K);
        int b, i, off, nib;
        matrix_row_to_band(a.kind, a.N, n, b, i);
        code_position(i, k, off, nib);
        const uint8_t *band = a.packed + (size_t)b * bb;
        const uint32_t word = *reinterpret_cast<const uint32_t *>(band + (off & ~3));
        const uint32_t reg = decode_reg(word, off & 3);
        const __half2 hh = *reinterpret_cast<const __half2 *>(&reg);
        const float code_val = nib ? __high2float(hh) : __low2float(hh);
        const uint32_t sb = band[scale_position(i, k / 16)];
        const float sc = e4m3x2_to_float2(sb).x;
        a.out[o] = code_val * sc * a.tscale;
    }
}

cudaError_t launch_pack(const PackArgs &a, cudaStream_t s)
{
    pack_kernel<<<1184, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_unpack(const UnpackArgs &a, cudaStream_t s)
{
    unpack_kernel<<<1184, 256, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_dequant(const DequantArgs &a, cudaStream_t s)
{
    dequant_kernel<<<1184, 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace moe
