// HBM-bound kernels of the ring-attention step:
//   K4 merge_lse     -- n-way log-sum-exp merge of partial attention results
//                       ("merge attention operation", "Ring Attention
//                       Algorithms" in "Context Parallelism for Scalable
//                       Million-Token Inference")
//   K5 permute_rows  -- natural <-> rank-major token order ("Load Balancing
//                       in CP": two chunks per rank)
//   K3 bwd_preprocess-- delta = rowsum(dO * O) for the softmax backward
//   zero_f32         -- clears fp32 gradient accumulators
//   bf16_to_f16      -- exact fp16 copies of the backward's bf16 operands
// All use 16-byte vector accesses with consecutive threads on consecutive
// addresses.
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"

namespace cpa {
namespace {

constexpr float kLog2e = 1.44269504088896340736f;
constexpr float kLn2 = 0.69314718055994530942f;

// Four consecutive elements of an O part (fp32 or bf16) as fp32.
__device__ __forceinline__ float4 load4(const float* __restrict__ base, int64_t off) {
  return __ldg(reinterpret_cast<const float4*>(base + off));
}
__device__ __forceinline__ float4 load4(const __nv_bfloat16* __restrict__ base, int64_t off) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(base + off));
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

// One warp per (row, head). Lane l handles float4 chunks l, l+32, ...
// TP: element type of the O parts (float or __nv_bfloat16).
template <int CHUNKS, typename TP>  // float4 chunks per lane (d/4/32 rounded up)
__global__ void __launch_bounds__(256) merge_lse_kernel(
    int n_parts, int64_t rows, int heads, int d, const TP* __restrict__ o_parts,
    int64_t part_stride, const float* __restrict__ lse_parts, int64_t lse_part_stride,
    __nv_bfloat16* __restrict__ o_out, float* __restrict__ o_out_f32,
    float* __restrict__ lse_out) {
  const int64_t wid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= rows * heads) return;
  const int64_t row = wid / heads;
  const int h = static_cast<int>(wid % heads);
  const int64_t lse_idx = static_cast<int64_t>(h) * rows + row;
  // M = max_i LSE_i (base 2)
  float M = -INFINITY;
  for (int i = lane; i < n_parts; i += 32)
    M = fmaxf(M, __ldg(lse_parts + i * lse_part_stride + lse_idx) * kLog2e);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const int n4 = d >> 2;
  float4 acc[CHUNKS];
#pragma unroll
  for (int c = 0; c < CHUNKS; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = -INFINITY;
  if (M != -INFINITY) {
    float S = 0.f;
    for (int i = lane; i < n_parts; i += 32)
      S += ptx::ex2(__ldg(lse_parts + i * lse_part_stride + lse_idx) * kLog2e - M);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
    L = M + ptx::lg2(S);
    const int64_t o_off = (row * heads + h) * static_cast<int64_t>(d);
    for (int i = 0; i < n_parts; ++i) {
      const float w = ptx::ex2(__ldg(lse_parts + i * lse_part_stride + lse_idx) * kLog2e - L);
      if (w == 0.f) continue;  // empty part (LSE = -inf) or negligible
#pragma unroll
      for (int c = 0; c < CHUNKS; ++c) {
        const int j = lane + 32 * c;
        if (j < n4) {
          const float4 v = load4(o_parts, i * part_stride + o_off + 4 * j);
          acc[c].x = fmaf(w, v.x, acc[c].x);
          acc[c].y = fmaf(w, v.y, acc[c].y);
          acc[c].z = fmaf(w, v.z, acc[c].z);
          acc[c].w = fmaf(w, v.w, acc[c].w);
        }
      }
    }
  }
  const int64_t o_off = (row * heads + h) * static_cast<int64_t>(d);
#pragma unroll
  for (int c = 0; c < CHUNKS; ++c) {
    const int j = lane + 32 * c;
    if (j < n4) {
      if (o_out_f32) reinterpret_cast<float4*>(o_out_f32 + o_off)[j] = acc[c];
      if (o_out) {
        uint2 pk;
        pk.x = ptx::pack_bf16(acc[c].x, acc[c].y);
        pk.y = ptx::pack_bf16(acc[c].z, acc[c].w);
        reinterpret_cast<uint2*>(o_out + o_off)[j] = pk;
      }
    }
  }
  if (lane == 0) lse_out[lse_idx] = (M == -INFINITY) ? -INFINITY : L * kLn2;
}

// The same merge for few (row, head) pairs and many parts (a decode row
// merges every rank's and every run's partial): one block of 16 warps per
// (row, head). The block first turns every part's LSE into its weight
// 2^(LSE_i - L), L = M + log2 sum_i 2^(LSE_i - M), in shared memory (one
// parallel pass for M, one for the sum); then each warp streams its share of
// the parts' rows (a float4 of d <= 128 per lane), up to sixteen loads in
// flight, and warp 0 adds the sixteen sums. A part whose weight is 0 (no
// visible key, or LSE = -inf) is neither loaded nor added. The block reads
// all parts before it writes, so o_out_f32 may alias part 0.
constexpr int kWideWarps = 16;
constexpr int kWideMaxParts = 4096;

// U: loads in flight per lane (4, 8 or 16); TP: element type of the O parts.
// The kernel waits on the previous kernel of the stream (programmatic
// dependent launch) before it reads anything.
template <int U, typename TP>
__global__ void __launch_bounds__(32 * kWideWarps) merge_lse_wide_kernel(
    int n_parts, int64_t rows, int heads, int d, const TP* __restrict__ o_parts,
    int64_t part_stride, const float* __restrict__ lse_parts, int64_t lse_part_stride,
    __nv_bfloat16* __restrict__ o_out, float* __restrict__ o_out_f32,
    float* __restrict__ lse_out) {
  __shared__ float s_w[kWideMaxParts];
  __shared__ float s_red[2][kWideWarps];
  __shared__ float4 s_acc[kWideWarps][32];
  ptx::grid_dep_wait();
  const int64_t pair = blockIdx.x;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t row = pair / heads;
  const int h = static_cast<int>(pair % heads);
  const int64_t lse_idx = static_cast<int64_t>(h) * rows + row;
  // the parts' LSEs (base 2) and their maximum
  float M = -INFINITY;
  for (int i = threadIdx.x; i < n_parts; i += 32 * kWideWarps) {
    const float x = __ldg(lse_parts + i * lse_part_stride + lse_idx) * kLog2e;
    s_w[i] = x;
    M = fmaxf(M, x);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  if (lane == 0) s_red[0][warp] = M;
  __syncthreads();
  M = s_red[0][0];
#pragma unroll
  for (int w = 1; w < kWideWarps; ++w) M = fmaxf(M, s_red[0][w]);
  float L = -INFINITY;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const int64_t o_off = (row * heads + h) * static_cast<int64_t>(d);
  const bool has = lane < (d >> 2);
  if (M != -INFINITY) {  // uniform across the block
    float S = 0.f;
    for (int i = threadIdx.x; i < n_parts; i += 32 * kWideWarps) S += ptx::ex2(s_w[i] - M);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) S += __shfl_xor_sync(0xffffffffu, S, o);
    if (lane == 0) s_red[1][warp] = S;
    __syncthreads();
    S = 0.f;
#pragma unroll
    for (int w = 0; w < kWideWarps; ++w) S += s_red[1][w];
    L = M + ptx::lg2(S);
    // each thread rewrites only the entries it read, so no barrier is needed
    // between the reads above and these writes
    for (int i = threadIdx.x; i < n_parts; i += 32 * kWideWarps) s_w[i] = ptx::ex2(s_w[i] - L);
    __syncthreads();
    // A warp's loads depend only on the weights (the same for its 32 lanes),
    // so a weight-0 part costs no load; a lane past d/4 reads chunk 0 (in
    // bounds) and its sum is not stored.
    const int l4 = has ? lane : 0;
    for (int i0 = warp; i0 < n_parts; i0 += kWideWarps * U) {
      float w[U];
      float4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * kWideWarps;
        w[u] = i < n_parts ? s_w[i] : 0.f;
        v[u] = w[u] != 0.f ? load4(o_parts, i * part_stride + o_off + 4 * l4)
                           : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        acc.x = fmaf(w[u], v[u].x, acc.x);
        acc.y = fmaf(w[u], v[u].y, acc.y);
        acc.z = fmaf(w[u], v[u].z, acc.z);
        acc.w = fmaf(w[u], v[u].w, acc.w);
      }
    }
  }
  s_acc[warp][lane] = acc;
  __syncthreads();
  if (warp == 0) {
    float4 t = s_acc[0][lane];
#pragma unroll
    for (int w = 1; w < kWideWarps; ++w) {
      const float4 u = s_acc[w][lane];
      t.x += u.x;
      t.y += u.y;
      t.z += u.z;
      t.w += u.w;
    }
    if (has) {
      if (o_out_f32) reinterpret_cast<float4*>(o_out_f32 + o_off)[lane] = t;
      if (o_out) {
        uint2 pk;
        pk.x = ptx::pack_bf16(t.x, t.y);
        pk.y = ptx::pack_bf16(t.z, t.w);
        reinterpret_cast<uint2*>(o_out + o_off)[lane] = pk;
      }
    }
    if (lane == 0) lse_out[lse_idx] = (M == -INFINITY) ? -INFINITY : L * kLn2;
  }
}

// out[dst] = in[src] for 16-byte vectors; row_map[i] = natural row of
// rank-major row i. to_natural: out[row_map[i]] = in[i]; else
// out[i] = in[row_map[i]].
__global__ void __launch_bounds__(256) permute_rows_kernel(const int32_t* __restrict__ row_map,
                                                           int64_t rows, int64_t vec_per_row,
                                                           int to_natural,
                                                           const uint4* __restrict__ in,
                                                           uint4* __restrict__ out) {
  const int64_t total = rows * vec_per_row;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t i = idx / vec_per_row;
    const int64_t v = idx - i * vec_per_row;
    const int64_t nat = __ldg(row_map + i);
    if (to_natural) out[nat * vec_per_row + v] = __ldg(in + i * vec_per_row + v);
    else out[i * vec_per_row + v] = __ldg(in + nat * vec_per_row + v);
  }
}

// K7 sequence <-> head all-to-all. Split: element (t, h, x) of [rows][heads]
// [vec] moves to sub-rank u = h / hs at [u][t][h % hs][x] (hs = heads / a2a);
// gather is the inverse. One 16-byte vector per thread, grid-stride; reads
// (split) or writes (gather) walk the source/destination rows in order, and
// every head row of `vec` vectors stays contiguous on both sides.
__global__ void __launch_bounds__(256) head_a2a_kernel(int64_t rows, int heads, int hs,
                                                       int64_t vec, int gather,
                                                       const uint4* __restrict__ in,
                                                       uint4* __restrict__ out) {
  const int64_t total = rows * heads * vec;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    // idx enumerates the [rows][heads][vec] side
    const int64_t x = idx % vec;
    const int64_t th = idx / vec;
    const int h = static_cast<int>(th % heads);
    const int64_t t = th / heads;
    const int u = h / hs;
    const int64_t other = ((static_cast<int64_t>(u) * rows + t) * hs + (h - u * hs)) * vec + x;
    if (gather) out[idx] = __ldg(in + other);
    else out[other] = __ldg(in + idx);
  }
}

// delta[h][t] = sum_x dO[t,h,x] * O[t,h,x], one warp per (t, h); lanes read
// 4 elements at a time. O is bf16 or fp32.
template <typename OT>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(int64_t rows, int heads, int d,
                                                             const OT* __restrict__ o,
                                                             const __nv_bfloat16* __restrict__ dout,
                                                             float* __restrict__ delta) {
  const int64_t wid = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wid >= rows * heads) return;
  const int64_t t = wid / heads;
  const int h = static_cast<int>(wid % heads);
  const int64_t off = wid * d;  // (t*heads + h)*d
  float acc = 0.f;
  for (int x = lane * 4; x < d; x += 128) {
    float fo[4];
    if constexpr (sizeof(OT) == 4) {
      const float4 a = __ldg(reinterpret_cast<const float4*>(o + off + x));
      fo[0] = a.x; fo[1] = a.y; fo[2] = a.z; fo[3] = a.w;
    } else {
      const uint2 a = __ldg(reinterpret_cast<const uint2*>(o + off + x));
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
      const float2 f0 = __bfloat1622float2(a2[0]), f1 = __bfloat1622float2(a2[1]);
      fo[0] = f0.x; fo[1] = f0.y; fo[2] = f1.x; fo[3] = f1.y;
    }
    const uint2 b = __ldg(reinterpret_cast<const uint2*>(dout + off + x));
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
    const float2 g0 = __bfloat1622float2(b2[0]), g1 = __bfloat1622float2(b2[1]);
    acc = fmaf(fo[0], g0.x, acc);
    acc = fmaf(fo[1], g0.y, acc);
    acc = fmaf(fo[2], g1.x, acc);
    acc = fmaf(fo[3], g1.y, acc);
  }
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  if (lane == 0) delta[static_cast<int64_t>(h) * rows + t] = acc;
}

__global__ void __launch_bounds__(256) zero_f32_kernel(float4* __restrict__ p, int64_t n4,
                                                       float* __restrict__ tail, int n_tail) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    p[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (blockIdx.x == 0 && threadIdx.x < n_tail) tail[threadIdx.x] = 0.f;
}

// 8 values per thread. bf16 values in [2^-14, 65504] convert exactly; a
// finite value above 65504 records CP_ATTN_ERR_RANGE in the status word.
__global__ void __launch_bounds__(256) bf16_to_f16_kernel(const uint4* __restrict__ in,
                                                          uint4* __restrict__ out, int64_t n8,
                                                          int32_t* status) {
  bool bad = false;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint4 a = __ldg(in + i);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    uint4 r;
    uint32_t* rr = reinterpret_cast<uint32_t*>(&r);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(b2[k]);
      bad |= (fabsf(f.x) > 65504.f && fabsf(f.x) <= 3.4e38f) ||
             (fabsf(f.y) > 65504.f && fabsf(f.y) <= 3.4e38f);
      rr[k] = ptx::pack_f16(f.x, f.y);
    }
    out[i] = r;
  }
  if (bad) atomicCAS(status, 0, static_cast<int>(CP_ATTN_ERR_RANGE));
}

// K6 finalize of bf16 gradients: 8 fp32 values per thread -> bf16, rounded
// to nearest even (grid-stride; 32 bytes read, 16 written per thread and
// iteration).
__global__ void __launch_bounds__(256) f32_to_bf16_kernel(const float4* __restrict__ in,
                                                          uint4* __restrict__ out, int64_t n8) {
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 a = __ldg(in + 2 * i);
    const float4 b = __ldg(in + 2 * i + 1);
    out[i] = make_uint4(ptx::pack_bf16(a.x, a.y), ptx::pack_bf16(a.z, a.w),
                        ptx::pack_bf16(b.x, b.y), ptx::pack_bf16(b.z, b.w));
  }
}

// One CTA waits on an mbarrier that nothing arrives on; the bounded wait
// gives up after limit_ns and records the timeout like every kernel wait.
__global__ void selftest_wait_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bar), 1);
    abort_flag = 0;
    ptx::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 &&
      !ptx::mbar_wait(ptx::smem_u32(&bar), 0, &abort_flag, limit_ns))
    ptx::record_timeout(status, &abort_flag, 0xdead);
}

int grid_for(int64_t work, int per_block, int cap) {
  const int64_t g = (work + per_block - 1) / per_block;
  return static_cast<int>(g < 1 ? 1 : (g > cap ? cap : g));
}

cp_attn_status check_launch(const char* what) {
  const cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return fail(CP_ATTN_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(err));
  count_launch();
  return CP_ATTN_OK;
}

}  // namespace

cp_attn_status launch_bf16_to_f16(const void* in, void* out, int64_t n, int32_t* status,
                                  cudaStream_t s) {
  const int64_t n8 = n / 8;
  if (n8 == 0) return CP_ATTN_OK;
  bf16_to_f16_kernel<<<grid_for(n8, 256, 152 * 16), 256, 0, s>>>(
      static_cast<const uint4*>(in), static_cast<uint4*>(out), n8, status);
  return check_launch("bf16_to_f16");
}

cp_attn_status launch_f32_to_bf16(const float* in, void* out, int64_t n, cudaStream_t s) {
  const int64_t n8 = n / 8;
  if (n8 == 0) return CP_ATTN_OK;
  f32_to_bf16_kernel<<<grid_for(n8, 256, 152 * 16), 256, 0, s>>>(
      reinterpret_cast<const float4*>(in), static_cast<uint4*>(out), n8);
  return check_launch("f32_to_bf16");
}

cp_attn_status launch_selftest_wait(int32_t* status, uint64_t limit_ns, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return check_launch("selftest_wait");
}

namespace {

template <typename TP>
cp_attn_status merge_lse_typed(int n_parts, int64_t rows, int heads, int d, const TP* o_parts,
                               int64_t part_stride, const float* lse_parts,
                               int64_t lse_part_stride, __nv_bfloat16* o_out, float* o_out_f32,
                               float* lse_out, cudaStream_t s, bool pdl) {
  const int64_t warps = rows * heads;
  if (warps == 0) return CP_ATTN_OK;
  // few (row, head) pairs with many parts: a block of warps per pair
  if (d <= 128 && n_parts >= 16 && n_parts <= kWideMaxParts && warps * kWideWarps <= 152 * 64) {
    const int per_warp = (n_parts + kWideWarps - 1) / kWideWarps;
    auto kernel = per_warp <= 4   ? merge_lse_wide_kernel<4, TP>
                  : per_warp <= 8 ? merge_lse_wide_kernel<8, TP>
                                  : merge_lse_wide_kernel<16, TP>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(warps));
    cfg.blockDim = dim3(32 * kWideWarps);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    const cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, n_parts, rows, heads, d, o_parts,
                                               part_stride, lse_parts, lse_part_stride, o_out,
                                               o_out_f32, lse_out);
    if (err != cudaSuccess) {
      cudaGetLastError();
      return fail(CP_ATTN_ERR_CUDA, std::string("merge_lse: ") + cudaGetErrorString(err));
    }
    return check_launch("merge_lse");
  }
  const int64_t blocks = (warps * 32 + 255) / 256;
  if (d <= 128)
    merge_lse_kernel<1, TP><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        n_parts, rows, heads, d, o_parts, part_stride, lse_parts, lse_part_stride, o_out,
        o_out_f32, lse_out);
  else
    merge_lse_kernel<2, TP><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        n_parts, rows, heads, d, o_parts, part_stride, lse_parts, lse_part_stride, o_out,
        o_out_f32, lse_out);
  return check_launch("merge_lse");
}

}  // namespace

cp_attn_status launch_merge_lse(int n_parts, int64_t rows, int heads, int d,
                                const void* o_parts, int64_t part_stride,
                                const float* lse_parts, int64_t lse_part_stride,
                                __nv_bfloat16* o_out, float* o_out_f32, float* lse_out,
                                cudaStream_t s, bool parts_bf16, bool pdl) {
  if (parts_bf16)
    return merge_lse_typed(n_parts, rows, heads, d, static_cast<const __nv_bfloat16*>(o_parts),
                           part_stride, lse_parts, lse_part_stride, o_out, o_out_f32, lse_out, s,
                           pdl);
  return merge_lse_typed(n_parts, rows, heads, d, static_cast<const float*>(o_parts), part_stride,
                         lse_parts, lse_part_stride, o_out, o_out_f32, lse_out, s, pdl);
}

cp_attn_status launch_permute_rows(const int32_t* row_map, int64_t rows, int64_t row_bytes,
                                   int to_natural, const void* in, void* out, cudaStream_t s) {
  const int64_t vpr = row_bytes / 16;
  if (rows * vpr == 0) return CP_ATTN_OK;
  permute_rows_kernel<<<grid_for(rows * vpr, 256, 152 * 16), 256, 0, s>>>(
      row_map, rows, vpr, to_natural, static_cast<const uint4*>(in), static_cast<uint4*>(out));
  return check_launch("permute_rows");
}

cp_attn_status launch_head_a2a(int64_t rows, int heads, int64_t head_bytes, int a2a, int gather,
                               const void* in, void* out, cudaStream_t s) {
  const int64_t vec = head_bytes / 16;
  const int64_t total = rows * heads * vec;
  if (total == 0) return CP_ATTN_OK;
  head_a2a_kernel<<<grid_for(total, 256, 152 * 16), 256, 0, s>>>(
      rows, heads, heads / a2a, vec, gather, static_cast<const uint4*>(in),
      static_cast<uint4*>(out));
  return check_launch("head_a2a");
}

cp_attn_status launch_bwd_preprocess(int64_t rows, int heads, int d, const __nv_bfloat16* o,
                                     const float* o_f32, const __nv_bfloat16* dout,
                                     float* delta, cudaStream_t s) {
  const int64_t warps = rows * heads;
  if (warps == 0) return CP_ATTN_OK;
  const int64_t blocks = (warps * 32 + 255) / 256;
  if (o_f32)
    bwd_preprocess_kernel<float><<<static_cast<unsigned>(blocks), 256, 0, s>>>(rows, heads, d,
                                                                               o_f32, dout, delta);
  else
    bwd_preprocess_kernel<__nv_bfloat16><<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        rows, heads, d, o, dout, delta);
  return check_launch("bwd_preprocess");
}

cp_attn_status launch_zero_f32(float* p, int64_t n, cudaStream_t s) {
  if (n == 0) return CP_ATTN_OK;
  const int64_t n4 = n / 4;
  const int n_tail = static_cast<int>(n - n4 * 4);
  zero_f32_kernel<<<grid_for(n4 > 0 ? n4 : 1, 256, 152 * 16), 256, 0, s>>>(
      reinterpret_cast<float4*>(p), n4, p + n4 * 4, n_tail);
  return check_launch("zero_f32");
}

}  // namespace cpa
