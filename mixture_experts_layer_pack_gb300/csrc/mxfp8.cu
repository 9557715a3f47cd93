// MXFP8 quantisation (OCP MX v1.0: E4M3 elements, one E8M0 shared exponent
// per 32 consecutive elements) and the weight-scale swizzle into the layout
// the block-scaled tensor-core MMA reads.
//
// "feat(moe): add a megakernel backend with MOK integration", Supported
// configurations (MXFP8 routed experts) and Design > MCore-owned parameters
// (converted scale layouts refreshed once per optimizer iteration at stable
// addresses); "Add Mixture-of-Kittens MoE backend on main", review threads on
// _swizzle_mxfp8_scale (rowwise and columnwise compact E8M0 scales converted
// to the GEMM's swizzled layout; columnwise scale shape (rows // 32, columns)).
#include "../../include/moe.h"
#include "device_common.cuh"
#include "internal.h"

namespace moe {

namespace {

// blocks of 32 along each row; a lane owns 8 consecutive elements, 4 lanes a block
__global__ void __launch_bounds__(256) quant_rows_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows, int cols,
                                                         int64_t ld, uint8_t* __restrict__ q, int64_t ldq,
                                                         uint8_t* __restrict__ scales) {
    const int vecs = cols / 8;
    const int64_t total = rows * vecs;
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
    for (int64_t base = ((int64_t(blockIdx.x) * blockDim.x + threadIdx.x) >> 5) * 32; base < total;
         base += nwarps * 32) {
        const int64_t i = base + lane;
        const bool active = i < total;
        const int64_t row = active ? i / vecs : 0;
        const int v = active ? int(i - row * vecs) : 0;
        float f[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (active) {
            const uint4 w = __ldg(reinterpret_cast<const uint4*>(x + row * ld) + v);
            unpack_bf16x2(w.x, f[0], f[1]);
            unpack_bf16x2(w.y, f[2], f[3]);
            unpack_bf16x2(w.z, f[4], f[5]);
            unpack_bf16x2(w.w, f[6], f[7]);
        }
        float amax = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(f[j]));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        const uint32_t code = e8m0_code(amax);
        const float mul = e8m0_inv_scale(code);
        if (active) {
            uint2 out;
            out.x = e4m3x4(f[0] * mul, f[1] * mul, f[2] * mul, f[3] * mul);
            out.y = e4m3x4(f[4] * mul, f[5] * mul, f[6] * mul, f[7] * mul);
            *reinterpret_cast<uint2*>(q + row * ldq + int64_t(v) * 8) = out;
            if ((lane & 3) == 0) scales[row * (cols / 32) + v / 4] = uint8_t(code);
        }
    }
}

// blocks of 32 down each column; a thread owns one (32-row block, column)
__global__ void __launch_bounds__(256) quant_cols_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows, int cols,
                                                         int64_t ld, uint8_t* __restrict__ q, int64_t ldq,
                                                         uint8_t* __restrict__ scales) {
    const int64_t total = (rows / 32) * cols;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t rb = i / cols;
        const int c = int(i - rb * cols);
        const __nv_bfloat16* src = x + rb * 32 * ld + c;
        float f[32];
        float amax = 0.0f;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            f[r] = __bfloat162float(src[int64_t(r) * ld]);
            amax = fmaxf(amax, fabsf(f[r]));
        }
        const uint32_t code = e8m0_code(amax);
        const float mul = e8m0_inv_scale(code);
        uint8_t* dst = q + rb * 32 * ldq + c;
#pragma unroll
        for (int r = 0; r < 32; ++r)
            dst[int64_t(r) * ldq] = __nv_cvt_float_to_fp8(f[r] * mul, __NV_SATFINITE, __NV_E4M3);
        scales[rb * cols + c] = uint8_t(code);
    }
}

// Swizzle of compact E8M0 weight scales into per-expert scale-factor atoms
// [E][n_tiles][k_blocks/4][512 B]. Row n of N-tile nt and K block kb come from:
//   SW_ROW      src0[e][nt*128 + n][kb]                       (row scales, K along the row)
//   SW_ROW_GU   rows 0..63 of a tile: gate row nt*64 + n, rows 64..127: up row nt*64 + n - 64
//   SW_COL      src0[e][kb][nt*128 + n]                       (column scales: K runs down the rows)
//   SW_COL_GU   kb < kb_split: gate src0[e][kb][..], else up src1[e][kb - kb_split][..]
enum SwizzleMode : int { SW_ROW = 0, SW_ROW_GU = 1, SW_COL = 2, SW_COL_GU = 3 };

// tab0 / tab1: device arrays of the E experts' source bases
__global__ void __launch_bounds__(256) swizzle_scales_kernel(int mode, const uint8_t* const* __restrict__ tab0,
                                                             const uint8_t* const* __restrict__ tab1,
                                                             int64_t src_rs, int E, int n_tiles, int k_blocks,
                                                             int kb_split, uint8_t* __restrict__ dst) {
    const int64_t per_expert = int64_t(n_tiles) * k_blocks * 128;
    const int64_t total = per_expert * E;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int e = int(i / per_expert);
        int64_t rem = i - e * per_expert;
        const int nt = int(rem / (int64_t(k_blocks) * 128));
        rem -= int64_t(nt) * k_blocks * 128;
        const int kb = int(rem / 128);
        const int n = int(rem - int64_t(kb) * 128);
        const uint8_t* src0 = tab0[e];
        uint8_t v;
        if (mode == SW_ROW) {
            v = src0[int64_t(nt * 128 + n) * src_rs + kb];
        } else if (mode == SW_ROW_GU) {
            const uint8_t* s = n < 64 ? src0 : tab1[e];
            v = s[int64_t(nt * 64 + (n & 63)) * src_rs + kb];
        } else if (mode == SW_COL) {
            v = src0[int64_t(kb) * src_rs + nt * 128 + n];
        } else {
            v = kb < kb_split ? src0[int64_t(kb) * src_rs + nt * 128 + n]
                              : tab1[e][int64_t(kb - kb_split) * src_rs + nt * 128 + n];
        }
        dst[e * per_expert + sf_atom_offset(int64_t(nt) * 128 + n, kb, k_blocks) - int64_t(nt) * 0] = v;
    }
}

int grid_for(int64_t work, int threads) {
    int64_t g = (work + threads - 1) / threads;
    if (g > 65535) g = 65535;
    return g < 1 ? 1 : int(g);
}

}  // namespace

cudaError_t launch_swizzle_scales(int mode, const uint8_t* const* tab0, const uint8_t* const* tab1, int64_t src_rs,
                                  int E, int n_tiles, int k_blocks, int kb_split, uint8_t* dst, cudaStream_t st) {
    const int64_t total = int64_t(E) * n_tiles * k_blocks * 128;
    swizzle_scales_kernel<<<grid_for(total, 256), 256, 0, st>>>(mode, tab0, tab1, src_rs, E, n_tiles, k_blocks,
                                                                  kb_split, dst);
    count_launch();
    return cudaGetLastError();
}

}  // namespace moe

extern "C" moe_status moe_quantize_mxfp8(const void* x, int64_t rows, int64_t cols, int64_t ld, int32_t axis,
                                         uint8_t* q, int64_t ldq, uint8_t* scales, void* stream) {
    using namespace moe;
    if (rows < 0 || cols <= 0 || ld < cols || ldq < cols || (axis != 0 && axis != 1)) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!x || !q || !scales) return MOE_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (axis == 1) {
        if (cols % 32 || ld % 8 || ldq % 8 || (reinterpret_cast<uintptr_t>(x) & 15) ||
            (reinterpret_cast<uintptr_t>(q) & 7))
            return MOE_ERR_INVALID_ARG;
        const int64_t work = rows * (cols / 8);
        quant_rows_kernel<<<grid_for(work, 256), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(x), rows, int(cols),
                                                                ld, q, ldq, scales);
    } else {
        if (rows % 32) return MOE_ERR_INVALID_ARG;
        const int64_t work = (rows / 32) * cols;
        quant_cols_kernel<<<grid_for(work, 256), 256, 0, st>>>(static_cast<const __nv_bfloat16*>(x), rows, int(cols),
                                                                ld, q, ldq, scales);
    }
    count_launch();
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
