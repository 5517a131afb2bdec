// Per-tensor E4M3 quantization of the FP8 path ("Experimental Setup &
// Results" in "Context Parallelism for Scalable Million-Token Inference": the
// Llama 3 405B model of the benchmarks is quantized to FP8 throughout).
//
// With amax = max |x| over the tensor, an element is stored as
// RN-even(fp32(x) * fp32(448 / amax)) clamped to +-448, and stands for
// code * fp32(amax / 448); an all-zero tensor uses scale 1. E4M3 is the OCP
// 8-bit format: bias 7, three mantissa bits, largest finite value 448.
//   absmax_bf16       -- amax of a bf16 tensor (fp32 bits, atomic maximum)
//   quantize_rows     -- [rows][heads][d] bf16 -> the same layout in E4M3
//   quantize_t        -- [rows][heads][d] bf16 -> [heads][d][rows] E4M3, the
//                        K-major layout of V as the B operand of O = P V
// All three are HBM-bound: 16-byte loads, consecutive threads on consecutive
// addresses.
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"

namespace cpa {
namespace {

constexpr float kE4M3Max = 448.f;

__device__ __forceinline__ float quant_inv(const unsigned int* amax_bits) {
  const float a = __uint_as_float(__ldg(amax_bits));
  return a > 0.f ? kE4M3Max / a : 1.f;
}

__device__ __forceinline__ void write_scale(const unsigned int* amax_bits, float* scale) {
  if (scale && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    const float a = __uint_as_float(__ldg(amax_bits));
    *scale = a > 0.f ? a / kE4M3Max : 1.f;
  }
}

// Non-negative floats order like their bit patterns, so the maximum is an
// unsigned atomic maximum on the bits. NaN inputs are ignored (fmaxf).
__global__ void __launch_bounds__(256) absmax_bf16_kernel(const uint4* __restrict__ in, int64_t n8,
                                                          unsigned int* amax_bits) {
  float m = 0.f;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 a = __ldg(in + i);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&a);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(b2[k]);
      m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float s_m[8];
  if ((threadIdx.x & 31) == 0) s_m[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = s_m[0];
    for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) b = fmaxf(b, s_m[w]);
    atomicMax(amax_bits, __float_as_uint(b));
  }
}

// Eight values per thread per step: 16 bytes in, 8 bytes out.
__global__ void __launch_bounds__(256) quantize_rows_kernel(const uint4* __restrict__ in, int64_t n8,
                                                            const unsigned int* amax_bits,
                                                            uint2* __restrict__ out, float* scale) {
  write_scale(amax_bits, scale);
  const float inv = quant_inv(amax_bits);
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 a = __ldg(in + i);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    float f[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 t = __bfloat1622float2(b2[k]);
      f[2 * k] = t.x * inv;
      f[2 * k + 1] = t.y * inv;
    }
    out[i] = make_uint2(ptx::pack_e4m3x4(f[0], f[1], f[2], f[3]),
                        ptx::pack_e4m3x4(f[4], f[5], f[6], f[7]));
  }
}

// One block per (64 rows, head): the 64 x d tile is quantized into shared
// memory as [d][64] bytes, then written out as d rows of 64 contiguous bytes.
constexpr int kTRows = 64;
template <int D>
__global__ void __launch_bounds__(256) quantize_t_kernel(const __nv_bfloat16* __restrict__ in,
                                                         int64_t rows, int heads,
                                                         const unsigned int* amax_bits,
                                                         uint8_t* __restrict__ out, float* scale) {
  write_scale(amax_bits, scale);
  const float inv = quant_inv(amax_bits);
  __shared__ __align__(16) uint8_t tile[D][kTRows + 16];
  const int64_t r0 = static_cast<int64_t>(blockIdx.x) * kTRows;
  const int h = blockIdx.y;
  constexpr int kChunks = kTRows * D / 8;  // 8 values per chunk
  for (int c = threadIdx.x; c < kChunks; c += blockDim.x) {
    const int r = c / (D / 8);
    const int d0 = (c % (D / 8)) * 8;
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(
        in + ((r0 + r) * heads + h) * static_cast<int64_t>(D) + d0));
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&a);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 t = __bfloat1622float2(b2[k]);
      const uint32_t q = ptx::pack_e4m3x4(t.x * inv, t.y * inv, 0.f, 0.f);
      tile[d0 + 2 * k][r] = static_cast<uint8_t>(q & 0xFFu);
      tile[d0 + 2 * k + 1][r] = static_cast<uint8_t>((q >> 8) & 0xFFu);
    }
  }
  __syncthreads();
  // each thread writes 16 bytes (16 rows) of one d row
  constexpr int kVec = D * kTRows / 16;
  for (int c = threadIdx.x; c < kVec; c += blockDim.x) {
    const int dd = c / (kTRows / 16);
    const int rr = (c % (kTRows / 16)) * 16;
    *reinterpret_cast<uint4*>(out + (static_cast<int64_t>(h) * D + dd) * rows + r0 + rr) =
        *reinterpret_cast<const uint4*>(&tile[dd][rr]);
  }
}

cp_attn_status check(const char* what) {
  const cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return fail(CP_ATTN_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(err));
  count_launch();
  return CP_ATTN_OK;
}

unsigned grid_cap(int64_t work, int cap) {
  const int64_t g = (work + 255) / 256;
  return static_cast<unsigned>(g < 1 ? 1 : (g > cap ? cap : g));
}

}  // namespace

cp_attn_status launch_fp8_absmax(const void* x, int64_t n, unsigned int* amax_bits,
                                 cudaStream_t s) {
  const cudaError_t err = cudaMemsetAsync(amax_bits, 0, sizeof(unsigned int), s);
  if (err != cudaSuccess) return fail(CP_ATTN_ERR_CUDA, std::string("fp8_absmax memset: ") + cudaGetErrorString(err));
  const int64_t n8 = n / 8;
  if (n8 == 0) return CP_ATTN_OK;
  absmax_bf16_kernel<<<grid_cap(n8, 152 * 8), 256, 0, s>>>(static_cast<const uint4*>(x), n8,
                                                           amax_bits);
  return check("fp8_absmax");
}

cp_attn_status launch_fp8_quantize(const void* x, int64_t rows, int heads, int d,
                                   const unsigned int* amax_bits, int transpose, void* out,
                                   float* scale, cudaStream_t s) {
  const int64_t n8 = rows * heads * d / 8;
  if (n8 == 0) return CP_ATTN_OK;
  if (!transpose) {
    quantize_rows_kernel<<<grid_cap(n8, 152 * 16), 256, 0, s>>>(
        static_cast<const uint4*>(x), n8, amax_bits, static_cast<uint2*>(out), scale);
    return check("fp8_quantize");
  }
  const dim3 grid(static_cast<unsigned>(rows / kTRows), static_cast<unsigned>(heads));
  if (d == 128)
    quantize_t_kernel<128><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x), rows, heads,
                                                amax_bits, static_cast<uint8_t*>(out), scale);
  else
    quantize_t_kernel<64><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x), rows, heads,
                                               amax_bits, static_cast<uint8_t*>(out), scale);
  return check("fp8_quantize_t");
}

}  // namespace cpa
