// Device-side helpers shared by the MoE kernels: PTX wrappers for mbarriers,
// TMA (cp.async.bulk.tensor), tcgen05 (TMEM alloc, MMA, commit, loads) and the
// bounded waits every spin in this library goes through.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace moe {

// A wait longer than this is treated as a hang: the waiting kernel records
// kStatusTimeout and winds down instead of spinning on.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31; }

// ---------------------------------------------------------------- programmatic dependent launch
// Every kernel of the layer's forward and backward is launched with programmatic
// stream serialisation: it may start while its predecessor finishes, so it waits
// (griddepcontrol.wait: the predecessor has completed and its writes are
// visible) before its first global-memory access, then lets its own successor
// start launching.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase of `bar` with the given parity to complete. Gives up
// when another role of the CTA has aborted (*abort != 0) or after
// kWaitLimitNs; on a timeout it sets *abort and the timeout bit in *status.
// Returns false when it gave up.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            atomicOr(status, kStatusTimeout);
            return false;
        }
    }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_map(const void* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const void* map, uint64_t* bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const void* map, uint64_t* bar, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
        "[%5];" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// TMA store of a shared-memory box into global memory
__device__ __forceinline__ void tma_store_3d(const void* map, const void* src, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(z), "r"(smem_u32(src))
        : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// wait until at most N bulk groups of this thread are still reading shared memory
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// wait until at most N bulk groups of this thread are incomplete
template <int N>
__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// order this thread's generic-proxy shared-memory writes before later async-proxy (TMA) reads
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 inputs, fp32 accumulate)
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// arrive on `bar` once all previously issued tcgen05.mma of this thread complete
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// 32 lanes x 32 consecutive fp32 columns: thread i of the warp gets lane
// (base lane + i), columns [col, col+32)
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------- bf16 packing
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void unpack_bf16x2(uint32_t w, float& lo, float& hi) {
    __nv_bfloat162 v = *reinterpret_cast<__nv_bfloat162*>(&w);
    float2 f = __bfloat1622float2(v);
    lo = f.x;
    hi = f.y;
}

// 32 fp32 -> 32 bf16 stored as four 16-byte vectors (dst 16-byte aligned)
__device__ __forceinline__ void store_bf16x32(__nv_bfloat16* dst, const float (&v)[32]) {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 w;
        w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
        w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
        w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
        w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
        d[q] = w;
    }
}

__device__ __forceinline__ void store_f32x32(float* dst, const float (&v)[32]) {
    float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int q = 0; q < 8; ++q) d[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}

__device__ __forceinline__ void load_bf16x32(const __nv_bfloat16* src, float (&v)[32]) {
    const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 w = s[q];
        unpack_bf16x2(w.x, v[8 * q + 0], v[8 * q + 1]);
        unpack_bf16x2(w.y, v[8 * q + 2], v[8 * q + 3]);
        unpack_bf16x2(w.z, v[8 * q + 4], v[8 * q + 5]);
        unpack_bf16x2(w.w, v[8 * q + 6], v[8 * q + 7]);
    }
}

// ---------------------------------------------------------------- MXFP8 (OCP MX v1.0)
// Shared-exponent code of a 32-element block whose largest magnitude is amax:
// floor(log2 amax) - 8 (8 = largest E4M3 exponent) + 127, clamped to [0, 254];
// an all-zero block gets 0. For a normal fp32 amax floor(log2 amax) is its
// unbiased exponent, so the code is the biased exponent minus 8.
__device__ __forceinline__ uint32_t e8m0_code(float amax) {
    const int eb = int((__float_as_uint(amax) >> 23) & 0xFF);
    const int c = eb - 8;
    return uint32_t(c < 0 ? 0 : (c > 254 ? 254 : c));
}

// 2^(127 - code) as an fp32 (exact; code 254 gives the subnormal 2^-127)
__device__ __forceinline__ float e8m0_inv_scale(uint32_t code) {
    const int e = 254 - int(code);
    return e > 0 ? __uint_as_float(uint32_t(e) << 23) : __uint_as_float(0x00400000u);
}

// 2^(code - 127) as an fp32
__device__ __forceinline__ float e8m0_scale(uint32_t code) {
    return code > 0 ? __uint_as_float(code << 23) : __uint_as_float(0x00400000u);
}

// four fp32 -> four E4M3 codes (round to nearest even, saturating at +-448), first in the low byte
// (two paired conversions: the first value of each pair lands in the low byte)
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
    return uint32_t(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3)) |
           (uint32_t(__nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3)) << 16);
}

// value of an E4M3 code
__device__ __forceinline__ float e4m3_value(uint32_t code) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw(__nv_fp8_storage_t(code & 0xFF), __NV_E4M3);
    return __half2float(__half(h));
}

// Byte offset of the scale of (row r, 32-element K block kb) in the scale-factor
// layout the block-scaled MMA reads: per 128 rows x 4 K blocks one 512-byte atom,
// byte 16*(r%32) + 4*((r%128)/32) + kb%4; atoms ordered [r/128][kb/4].
__device__ __forceinline__ int64_t sf_atom_offset(int64_t r, int kb, int k_blocks) {
    return ((r >> 7) * (k_blocks >> 2) + (kb >> 2)) * 512 + 16 * (r & 31) + 4 * ((r & 127) >> 5) + (kb & 3);
}

// Warp-wide copy of one bf16 row (src null: zeros) that also writes its MXFP8
// quantisation along the row: a lane owns 8 consecutive elements (16 bytes), 4
// consecutive lanes one 32-element block. Each lane loads up to four vectors
// before it converts and stores any. vec_per_row = row length / 8 must be a
// multiple of 4; all 32 lanes must call it.
__device__ __forceinline__ void copy_quant_row(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                               uint8_t* __restrict__ q, uint8_t* __restrict__ sf, int64_t row,
                                               int vec_per_row) {
    constexpr int kInFlight = 4;
    const int lane = threadIdx.x & 31;
    const int k_blocks = vec_per_row / 4;
    uint8_t* qrow = q + row * int64_t(vec_per_row) * 8;
    for (int base = 0; base < vec_per_row; base += 32 * kInFlight) {
        uint4 w[kInFlight];
#pragma unroll
        for (int j = 0; j < kInFlight; ++j) {
            const int v = base + j * 32 + lane;
            w[j] = (src && v < vec_per_row) ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < kInFlight; ++j) {
            // a 4-lane block is active or idle as a whole: vec_per_row is a multiple of 4
            const int v = base + j * 32 + lane;
            float f[8];
            unpack_bf16x2(w[j].x, f[0], f[1]);
            unpack_bf16x2(w[j].y, f[2], f[3]);
            unpack_bf16x2(w[j].z, f[4], f[5]);
            unpack_bf16x2(w[j].w, f[6], f[7]);
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
            const uint32_t code = e8m0_code(amax);
            const float mul = e8m0_inv_scale(code);
            if (v < vec_per_row) {
                dst[v] = w[j];
                *reinterpret_cast<uint2*>(qrow + int64_t(v) * 8) =
                    make_uint2(e4m3x4(f[0] * mul, f[1] * mul, f[2] * mul, f[3] * mul),
                               e4m3x4(f[4] * mul, f[5] * mul, f[6] * mul, f[7] * mul));
                if ((lane & 3) == 0) sf[sf_atom_offset(row, v >> 2, k_blocks)] = uint8_t(code);
            }
        }
    }
}

// dst[0, n) = src[0, n) in 16-byte vectors (src null: zeros), by one warp: each lane
// has up to eight vectors in flight before it stores any
__device__ __forceinline__ void copy_row(const uint4* __restrict__ src, uint4* __restrict__ dst, int n) {
    const int lane = threadIdx.x & 31;
    for (int base = 0; base < n; base += 32 * 8) {
        uint4 w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int v = base + j * 32 + lane;
            w[j] = (src && v < n) ? __ldg(src + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int v = base + j * 32 + lane;
            if (v < n) dst[v] = w[j];
        }
    }
}

// SwiGLU pieces: silu(z) = z * sigmoid(z); d silu / dz = s (1 + z (1 - s))
// logistic function with the hardware reciprocal: a few ulp from the correctly rounded
// value; 0 where exp(-z) overflows
__device__ __forceinline__ float sigmoidf_(float z) { return __fdividef(1.0f, 1.0f + __expf(-z)); }

}  // namespace moe
