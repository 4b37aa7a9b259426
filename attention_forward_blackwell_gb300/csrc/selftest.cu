// Unit self-tests of the tcgen05 building blocks used by the prefill kernel.
//
// tmem_roundtrip: a no-op round trip through tensor memory (store, load,
// multiply by 1, store, load) must return its input bit for bit.
// "STAGE_D.md" reports that exactly this test failed in its 6-warp CuTeDSL
// kernel (load/store atoms with mismatched column mappings); here the load and
// the store use the same 32x32b shape, thread i <-> lane 32*(warp%4)+i.
//
// mma_tile: one 128x128 output tile through the same shared-memory layout,
// descriptors and instruction descriptors as the prefill kernel:
//   mode 0: D = A * B^T, A [128 x K] and B [128 x K] K-major (the score MMA,
//           issued as two N = 64 halves like the prefill kernel);
//   mode 1: D = P * V, P [128 x 128] placed in tensor memory as bf16 pairs,
//           V [128 keys x 128] MN-major in shared memory (the value MMA).
// The operands are staged into the 128-byte-swizzled layout with plain loads
// (16-byte granule g of row r lands at granule g ^ (r % 8)), the layout TMA
// produces with CU_TENSOR_MAP_SWIZZLE_128B.
#include "../../include/fa.h"
#include "common.cuh"
#include "ptx.cuh"

namespace fa {
namespace {

__global__ void __launch_bounds__(128) tmem_roundtrip_kernel(const float* in, float* out) {
    __shared__ uint32_t taddr_s;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = threadIdx.x;
    if (warp == 0) {
        tmem_alloc(smem_u32(&taddr_s), 64);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t t = taddr_s + ((uint32_t)(warp * 32) << 16);
    uint32_t v[32];
    for (int h = 0; h < 2; ++h) {
        for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(in[r * 64 + h * 32 + c]);
        tmem_st32(t + h * 32, v);
    }
    tmem_wait_st();
    for (int h = 0; h < 2; ++h) {
        tmem_ld32(t + h * 32, v);
        tmem_wait_ld();
        for (int c = 0; c < 32; ++c) v[c] = __float_as_uint(__uint_as_float(v[c]) * 1.0f);
        tmem_st32(t + h * 32, v);
    }
    tmem_wait_st();
    for (int h = 0; h < 2; ++h) {
        tmem_ld32(t + h * 32, v);
        tmem_wait_ld();
        for (int c = 0; c < 32; ++c) out[r * 64 + h * 32 + c] = __uint_as_float(v[c]);
    }
    (void)lane;
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(taddr_s, 64);
    }
}

// Copies a row-major bf16 matrix [rows x cols] (cols a multiple of 64) into
// 128-byte-swizzled 64-column chunks of `rows` x 128 bytes each.
__device__ void stage_sw128(uint8_t* smem, const uint16_t* g, int rows, int cols) {
    const int granules = rows * cols / 8;
    for (int e = threadIdx.x; e < granules; e += blockDim.x) {
        const int r = e / (cols / 8), gc = e % (cols / 8);
        const int chunk = gc / 8, gi = gc % 8;
        const uint4 val = *reinterpret_cast<const uint4*>(g + (size_t)r * cols + gc * 8);
        *reinterpret_cast<uint4*>(smem + chunk * rows * 128 + r * 128 + ((gi ^ (r & 7)) << 4)) = val;
    }
}

__global__ void __launch_bounds__(128) mma_tile_kernel(const uint16_t* a, const uint16_t* b,
                                                        float* d, int mode, int kdim,
                                                        unsigned int* err_word) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ uint32_t taddr_s;
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sA = smem_u32(smem);
    const uint32_t sB = sA + 128 * kdim * 2;
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&taddr_s), 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = taddr_s;
    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
    const int r = threadIdx.x;
    if (mode == 0) {
        stage_sw128(smem, a, 128, kdim);
        stage_sw128(smem + 128 * kdim * 2, b, 128, kdim);
    } else {
        // P row r -> tensor memory columns [128, 192) as bf16 pairs
        uint32_t pk[32];
        for (int h = 0; h < 2; ++h) {
            for (int c = 0; c < 32; ++c)
                pk[c] = (uint32_t)a[r * 128 + h * 64 + 2 * c] |
                        ((uint32_t)a[r * 128 + h * 64 + 2 * c + 1] << 16);
            tmem_st32(lane_base + 128 + h * 32, pk);
        }
        tmem_wait_st();
        stage_sw128(smem + 128 * kdim * 2, b, 128, 128);   // V [keys x dims]
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (threadIdx.x == 0) {
        if (mode == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, 64, false, false);
            for (int hf = 0; hf < 2; ++hf)
                for (int kk = 0; kk < kdim / 16; ++kk) {
                    const uint32_t aa = sA + (kk / 4) * 128 * 128 + (kk % 4) * 32;
                    const uint32_t bb = sB + (kk / 4) * 128 * 128 + hf * 64 * 128 + (kk % 4) * 32;
                    umma_ss(tmem + hf * 64, sdesc_sw128(aa, 16, 1024), sdesc_sw128(bb, 16, 1024),
                            idesc, kk > 0 ? 1u : 0u);
                }
        } else {
            constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false, true);
            for (int kk = 0; kk < 8; ++kk)
                umma_ts(tmem, tmem + 128 + kk * 8,
                        sdesc_sw128(sB + kk * 2048, 128 * 128, 1024), idesc, kk > 0 ? 1u : 0u);
        }
        tc_commit(smem_u32(&bar));
    }
    __syncwarp();
    const WaitCtx wc{smem_u32(&abort_flag), 1000000000u, err_word};
    const bool ok = mbar_wait(smem_u32(&bar), 0, wc, kErrWaitTimeout | 0xFEu);
    tc_fence_after();
    if (ok) {
        uint32_t v[32];
        for (int q = 0; q < 4; ++q) {
            tmem_ld32(lane_base + q * 32, v);
            tmem_wait_ld();
            for (int c = 0; c < 32; ++c) d[r * 128 + q * 32 + c] = __uint_as_float(v[c]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

__global__ void exp2_poly_kernel(const float* x, float* y, int n) {
    const int i = 2 * (blockIdx.x * blockDim.x + threadIdx.x);
    if (i + 1 < n) {
        const float2 r = exp2_poly_x2(make_float2(x[i], x[i + 1]));
        y[i] = r.x;
        y[i + 1] = r.y;
    } else if (i < n) {
        y[i] = exp2_poly_x2(make_float2(x[i], 0.f)).x;
    }
}

}  // namespace

cudaError_t launch_selftest_exp2_poly(const float* x, float* y, int n, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    const int threads = 256, pairs = (n + 1) / 2;
    exp2_poly_kernel<<<(pairs + threads - 1) / threads, threads, 0, s>>>(x, y, n);
    return cudaGetLastError();
}

cudaError_t launch_selftest_tmem_roundtrip(const float* in, float* out, cudaStream_t s) {
    tmem_roundtrip_kernel<<<1, 128, 0, s>>>(in, out);
    return cudaGetLastError();
}

cudaError_t launch_selftest_mma_tile(const uint16_t* a, const uint16_t* b, float* d, int mode,
                                     int kdim, unsigned int* err_word, cudaStream_t s) {
    const int smem = 1024 + 2 * 128 * (kdim > 128 ? kdim : 128) * 2;
    cudaError_t e = cudaFuncSetAttribute(mma_tile_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    mma_tile_kernel<<<1, 128, smem, s>>>(a, b, d, mode, kdim, err_word);
    return cudaGetLastError();
}

}  // namespace fa
