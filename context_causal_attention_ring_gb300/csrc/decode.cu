// K8: one-row decode over the emulated ring (Pass Q for decode).
//
// "Context Parallelism for Scalable Million-Token Inference", sections
// "Attention Compute Patterns in Multi-Turn Chat" (decode: the new token
// attends to every earlier token, a single-row attention) and "Ring
// Attention Algorithms" (Pass Q suits decode: the KV stays on its rank, the
// query visits every rank, each rank computes a partial attention of the row
// against its KV, and the partials are merged).
//
// One CTA computes the partial attention of one sequence's new row, for the
// G query heads of one KV head, against a run of L keys of one rank's shard
// (the shard is split further so that the grid fills the GPU). The work is
// bound by reading K and V once from HBM (2 * L * d * 2 bytes per CTA for
// G * L * d * 4 FLOP), so it runs on the CUDA cores, not the tensor cores:
//   1. scores s[j][h] = scale * q_h . k_j, K staged through shared memory in
//      64-key tiles (cp.async, double-buffered, 16-byte units XOR-swizzled
//      by row), one thread per (one or two keys, group of heads);
//   2. per head (half a warp each): max over the L keys, p = 2^(s - max),
//      sum;
//   3. O_h = sum_j p[j][h] v_j, V staged the same way, each warp taking 8
//      consecutive keys of a tile and each lane 4 (or 2) columns of d; the
//      warps' sums meet in shared memory;
//   4. O_h / l_h and LSE_h = ln l_h + max to the partial slots.
// The partials then go through the LSE merge (K4).
#include <cmath>
#include <cstring>

#include "kernels.h"
#include "ptx.cuh"

namespace cpa {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecTile = 64;    // keys per staged tile
constexpr int kDecMaxG = 16;    // query heads per KV head
constexpr int kDecMaxL = 512;   // keys per CTA
constexpr float kLn2d = 0.69314718055994530942f;
constexpr float kLog2ed = 1.44269504088896340736f;

struct DecParams {
  const __nv_bfloat16* q;  // [B][Hq][d]
  const __nv_bfloat16* k;  // [B][kv_len][Hkv][d]
  const __nv_bfloat16* v;
  float* o_part;           // [parts][B][Hq][d]
  float* lse_part;         // [parts][Hq][B]
  int B, Hq, Hkv, G;
  int64_t kv_len;
  int L;                   // keys per part (multiple of kDecTile, <= kDecMaxL)
  float scale_log2;        // softmax scale * log2(e)
};

template <int D>
struct DecSmem {
  static constexpr int kRowBytes = D * 2;
  static constexpr int kTileBytes = kDecTile * kRowBytes;
  static constexpr int kQ = 0;                                  // [kDecMaxG][D] f32
  static constexpr int kKV = kQ + kDecMaxG * D * 4;             // [2][kDecTile][D] bf16
  static constexpr int kS = kKV + 2 * kTileBytes;               // [kDecMaxG][kDecMaxL] f32
  static constexpr int kO = kS + kDecMaxL * kDecMaxG * 4;       // [kDecMaxG][D] f32
  static constexpr int kStat = kO + kDecMaxG * D * 4;           // max[G], sum[G]
  static constexpr int kBytes = kStat + 2 * kDecMaxG * 4;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src))
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Stage keys [key0, key0 + 64) of (sequence b, KV head kh) of `src` into a
// tile: row j at j * row bytes, 16-byte unit c at unit c ^ (j & 7).
template <int D>
__device__ __forceinline__ void stage_tile(uint32_t tile, const __nv_bfloat16* src,
                                           const DecParams& p, int b, int kh, int64_t key0) {
  constexpr int kUnits = D / 8;  // 16-byte units per row
  for (int i = threadIdx.x; i < kDecTile * kUnits; i += kDecThreads) {
    const int j = i / kUnits;
    const int c = i % kUnits;
    const __nv_bfloat16* g =
        src + ((static_cast<int64_t>(b) * p.kv_len + key0 + j) * p.Hkv + kh) * D + c * 8;
    cp_async16(tile + j * DecSmem<D>::kRowBytes + ((c ^ (j & 7)) << 4), g);
  }
  cp_async_commit();
}

template <int D, int HPG>  // HPG: query heads per thread-key in the score phase (1, 2, 4)
__global__ void __launch_bounds__(kDecThreads) decode_partial_kernel(const DecParams p) {
  using S = DecSmem<D>;
  extern __shared__ __align__(16) uint8_t smem[];
  float* q_s = reinterpret_cast<float*>(smem + S::kQ);
  float* s_s = reinterpret_cast<float*>(smem + S::kS);
  float* o_s = reinterpret_cast<float*>(smem + S::kO);
  float* st_max = reinterpret_cast<float*>(smem + S::kStat);
  float* st_sum = st_max + kDecMaxG;
  const uint32_t kv_s = ptx::smem_u32(smem + S::kKV);

  const int part = blockIdx.x;
  const int kh = blockIdx.y;
  const int b = blockIdx.z;
  const int t = threadIdx.x;
  const int warp = t >> 5;
  const int lane = t & 31;
  const int G = p.G;
  const int64_t key0 = static_cast<int64_t>(part) * p.L;
  const int n_tiles = p.L / kDecTile;

  stage_tile<D>(kv_s, p.k, p, b, kh, key0);
  // the group's query rows, pre-scaled to base-2 scores; O sums start at 0
  for (int i = t; i < kDecMaxG * D; i += kDecThreads) {
    const int h = i / D;
    float qv = 0.f;
    if (h < G)
      qv = __bfloat162float(p.q[(static_cast<int64_t>(b) * p.Hq + kh * G + h) * D + i % D]) *
           p.scale_log2;
    q_s[i] = qv;
    o_s[i] = 0.f;
  }

  // ---- 1. scores: thread = (KPT keys of the tile, group g of HPT heads).
  // KPT = 1 for up to 4 heads per group; 2 above, so that each 16-byte load
  // of K or of Q serves more FMAs.
  constexpr int KPT = HPG == 1 ? 1 : 2;
  constexpr int HPT = HPG == 1 ? 1 : HPG / 2;
  constexpr int kSlots = kDecTile / KPT;     // key slots per head group
  const int j0 = t % kSlots;
  const int g = t / kSlots;                  // a warp shares its group: Q reads broadcast
  for (int tile = 0; tile < n_tiles; ++tile) {
    if (tile + 1 < n_tiles) {
      stage_tile<D>(kv_s + ((tile + 1) & 1) * S::kTileBytes, p.k, p, b, kh,
                    key0 + (tile + 1) * kDecTile);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    float2 acc[KPT][HPT];
#pragma unroll
    for (int a2 = 0; a2 < KPT; ++a2)
#pragma unroll
      for (int i = 0; i < HPT; ++i) acc[a2][i] = make_float2(0.f, 0.f);
    const uint8_t* tb = smem + S::kKV + (tile & 1) * S::kTileBytes;
#pragma unroll 4
    for (int c = 0; c < D / 8; ++c) {
      float2 kf[KPT][4];
#pragma unroll
      for (int a2 = 0; a2 < KPT; ++a2) {
        const int j = j0 + a2 * kSlots;
        const uint4 kr = *reinterpret_cast<const uint4*>(tb + j * S::kRowBytes + ((c ^ (j & 7)) << 4));
        const __nv_bfloat162* k2 = reinterpret_cast<const __nv_bfloat162*>(&kr);
#pragma unroll
        for (int x = 0; x < 4; ++x) kf[a2][x] = __bfloat1622float2(k2[x]);
      }
#pragma unroll
      for (int i = 0; i < HPT; ++i) {
        const float4* qr = reinterpret_cast<const float4*>(q_s + (g * HPT + i) * D + c * 8);
        const float4 qa = qr[0], qb = qr[1];
#pragma unroll
        for (int a2 = 0; a2 < KPT; ++a2) {
          acc[a2][i] = ptx::fma2(make_float2(qa.x, qa.y), kf[a2][0], acc[a2][i]);
          acc[a2][i] = ptx::fma2(make_float2(qa.z, qa.w), kf[a2][1], acc[a2][i]);
          acc[a2][i] = ptx::fma2(make_float2(qb.x, qb.y), kf[a2][2], acc[a2][i]);
          acc[a2][i] = ptx::fma2(make_float2(qb.z, qb.w), kf[a2][3], acc[a2][i]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < HPT; ++i)
#pragma unroll
      for (int a2 = 0; a2 < KPT; ++a2)
        if (g * HPT + i < G)
          s_s[(g * HPT + i) * kDecMaxL + tile * kDecTile + j0 + a2 * kSlots] =
              acc[a2][i].x + acc[a2][i].y;
    __syncthreads();  // the tile buffer is reloaded two tiles on
  }
  // prefetch the first V tile while the softmax runs
  stage_tile<D>(kv_s, p.v, p, b, kh, key0);

  // ---- 2. per head: max, p = 2^(s - max), sum. Head h belongs to the 16
  // threads 16h .. 16h+15 (half a warp), each scanning every 16th key, so
  // both reductions stay inside the half-warp.
  {
    const int h = t >> 4;
    const int sub = t & 15;
    float* row = s_s + h * kDecMaxL;
    float m = -INFINITY;
    if (h < G)
      for (int k = sub; k < p.L; k += 16) m = fmaxf(m, row[k]);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float sum = 0.f;
    if (h < G)
      for (int k = sub; k < p.L; k += 16) {
        const float e = ptx::ex2(row[k] - m);
        row[k] = e;
        sum += e;
      }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (sub == 0 && h < G) {
      st_max[h] = m;
      st_sum[h] = sum;
    }
  }

  // ---- 3. O_h = sum_j p[j][h] v_j: warp takes every 8th key of a tile, lane
  // takes D/32 columns
  constexpr int kCols = D / 32;  // 4 (d = 128) or 2 (d = 64)
  float acc[kDecMaxG][kCols];
#pragma unroll
  for (int h = 0; h < kDecMaxG; ++h)
#pragma unroll
    for (int x = 0; x < kCols; ++x) acc[h][x] = 0.f;
  for (int tile = 0; tile < n_tiles; ++tile) {
    if (tile + 1 < n_tiles) {
      stage_tile<D>(kv_s + ((tile + 1) & 1) * S::kTileBytes, p.v, p, b, kh,
                    key0 + (tile + 1) * kDecTile);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const uint8_t* base = smem + S::kKV + (tile & 1) * S::kTileBytes;
    // warp w takes keys 8w .. 8w+7 of the tile: their p of one head are two
    // 16-byte loads (all lanes read the same address)
    constexpr int kKeysPerWarp = kDecTile / (kDecThreads / 32);
    float vf[kKeysPerWarp][kCols];
#pragma unroll
    for (int kk = 0; kk < kKeysPerWarp; ++kk) {
      const int jj = warp * kKeysPerWarp + kk;
      // this lane's kCols columns: byte offset lane*kCols*2 of the row
      const int off = lane * kCols * 2;
      const int unit = off >> 4;
      const uint8_t* src = base + jj * S::kRowBytes + (((unit ^ (jj & 7)) << 4) | (off & 15));
      if constexpr (kCols == 4) {
        const uint2 raw = *reinterpret_cast<const uint2*>(src);
        const __nv_bfloat162* v2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
        const float2 a = __bfloat1622float2(v2[0]), c = __bfloat1622float2(v2[1]);
        vf[kk][0] = a.x; vf[kk][1] = a.y; vf[kk][2] = c.x; vf[kk][3] = c.y;
      } else {
        const uint32_t raw = *reinterpret_cast<const uint32_t*>(src);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw));
        vf[kk][0] = a.x; vf[kk][1] = a.y;
      }
    }
    const float* pc = s_s + tile * kDecTile + warp * kKeysPerWarp;  // head h at h * kDecMaxL
#pragma unroll
    for (int h = 0; h < kDecMaxG; ++h) {
      if (h >= G) break;
      const float4 p0 = *reinterpret_cast<const float4*>(pc + h * kDecMaxL);
      const float4 p1 = *reinterpret_cast<const float4*>(pc + h * kDecMaxL + 4);
      const float ph[kKeysPerWarp] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
#pragma unroll
      for (int kk = 0; kk < kKeysPerWarp; ++kk)
#pragma unroll
        for (int x = 0; x < kCols; ++x) acc[h][x] = fmaf(ph[kk], vf[kk][x], acc[h][x]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int h = 0; h < kDecMaxG; ++h) {
    if (h >= G) break;
#pragma unroll
    for (int x = 0; x < kCols; ++x) atomicAdd(o_s + h * D + lane * kCols + x, acc[h][x]);
  }
  __syncthreads();

  // ---- 4. normalised partial O and its LSE
  const int64_t o_base = (static_cast<int64_t>(part) * p.B + b) * p.Hq + kh * G;
  for (int i = t; i < G * D; i += kDecThreads) {
    const int h = i / D;
    p.o_part[(o_base + h) * D + i % D] = o_s[i] / st_sum[h];
  }
  if (t < G)
    p.lse_part[(static_cast<int64_t>(part) * p.Hq + kh * G + t) * p.B + b] =
        (st_max[t] + ptx::lg2(st_sum[t])) * kLn2d;
}

// Keys per CTA: the largest of 512, 256, 128, 64 that divides the shard and
// still leaves about four CTAs per SM; 64 if none does.
int pick_part_len(int64_t shard, int64_t ctas_per_part) {
  const int64_t want = 152 * 4;
  for (int L : {kDecMaxL, 256, 128})
    if (shard % L == 0 && (shard / L) * ctas_per_part >= want) return L;
  return kDecTile;
}

cp_attn_status validate(const cp_attn_decode_desc* d) {
  if (!d) return fail(CP_ATTN_ERR_INVALID_ARG, "decode: null descriptor");
  if (d->batch <= 0 || d->cp <= 0 || d->kv_len <= 0)
    return fail(CP_ATTN_ERR_SHAPE, "decode: batch, cp and kv_len must be positive");
  if (d->head_dim != 64 && d->head_dim != 128)
    return fail(CP_ATTN_ERR_UNSUPPORTED, "decode: head_dim must be 64 or 128");
  if (d->n_kv_heads <= 0 || d->n_q_heads <= 0 || d->n_q_heads % d->n_kv_heads)
    return fail(CP_ATTN_ERR_SHAPE, "decode: n_q_heads must be a positive multiple of n_kv_heads");
  if (d->n_q_heads / d->n_kv_heads > kDecMaxG)
    return fail(CP_ATTN_ERR_UNSUPPORTED, "decode: at most 16 query heads per KV head");
  if (d->kv_len % (static_cast<int64_t>(d->cp) * kDecTile))
    return fail(CP_ATTN_ERR_SHAPE, "decode: kv_len must be a multiple of 64 * cp");
  if (!(d->softmax_scale >= 0.f) || std::isinf(d->softmax_scale))
    return fail(CP_ATTN_ERR_INVALID_ARG, "decode: softmax_scale must be finite and >= 0");
  return CP_ATTN_OK;
}

int64_t n_parts(const cp_attn_decode_desc* d) {
  const int64_t shard = d->kv_len / d->cp;
  const int L = pick_part_len(shard, static_cast<int64_t>(d->cp) * d->n_kv_heads * d->batch);
  return d->kv_len / L;
}

template <int D, int HPG>
cp_attn_status launch(const DecParams& p, int parts, cudaStream_t s) {
  const size_t smem = DecSmem<D>::kBytes;
  static bool attr = false;
  if (!attr) {
    const cudaError_t err = cudaFuncSetAttribute(decode_partial_kernel<D, HPG>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(smem));
    if (err != cudaSuccess)
      return fail(CP_ATTN_ERR_CUDA, std::string("decode attr: ") + cudaGetErrorString(err));
    attr = true;
  }
  decode_partial_kernel<D, HPG><<<dim3(parts, p.Hkv, p.B), kDecThreads, smem, s>>>(p);
  const cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return fail(CP_ATTN_ERR_CUDA, std::string("decode: ") + cudaGetErrorString(err));
  count_launch();
  return CP_ATTN_OK;
}

}  // namespace
}  // namespace cpa

extern "C" {

cp_attn_status cp_attn_decode_workspace_size(const cp_attn_decode_desc* desc, size_t* bytes) {
  cpa::clear_error();
  cp_attn_status st = cpa::validate(desc);
  if (st != CP_ATTN_OK) return st;
  if (!bytes) return cpa::fail(CP_ATTN_ERR_INVALID_ARG, "decode_workspace_size: null out");
  const int64_t parts = cpa::n_parts(desc);
  const int64_t rows = static_cast<int64_t>(desc->batch) * desc->n_q_heads;
  const size_t o_bytes = static_cast<size_t>(parts * rows * desc->head_dim) * 4;
  *bytes = ((o_bytes + 255) / 256) * 256 + static_cast<size_t>(parts * rows) * 4;
  return CP_ATTN_OK;
}

cp_attn_status cp_attn_decode(const cp_attn_decode_desc* desc, const void* q, const void* k,
                              const void* v, void* o, float* lse, void* workspace,
                              size_t workspace_bytes, void* stream) {
  cpa::clear_error();
  size_t need = 0;
  cp_attn_status st = cp_attn_decode_workspace_size(desc, &need);
  if (st != CP_ATTN_OK) return st;
  if (!q || !k || !v || !o || !lse || !workspace)
    return cpa::fail(CP_ATTN_ERR_INVALID_ARG, "decode: null pointer");
  for (const void* ptr : {q, k, v, static_cast<const void*>(o), static_cast<const void*>(lse),
                          static_cast<const void*>(workspace)})
    if (reinterpret_cast<uintptr_t>(ptr) % 16)
      return cpa::fail(CP_ATTN_ERR_INVALID_ARG, "decode: pointers must be 16-byte aligned");
  if (workspace_bytes < need)
    return cpa::fail(CP_ATTN_ERR_SHAPE, "decode: workspace too small");
  const int64_t parts = cpa::n_parts(desc);
  const int G = desc->n_q_heads / desc->n_kv_heads;
  const int64_t rows = static_cast<int64_t>(desc->batch) * desc->n_q_heads;
  const size_t o_bytes = static_cast<size_t>(parts * rows * desc->head_dim) * 4;
  float* o_part = static_cast<float*>(workspace);
  float* lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + ((o_bytes + 255) / 256) * 256);
  cpa::DecParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.k = static_cast<const __nv_bfloat16*>(k);
  p.v = static_cast<const __nv_bfloat16*>(v);
  p.o_part = o_part;
  p.lse_part = lse_part;
  p.B = desc->batch;
  p.Hq = desc->n_q_heads;
  p.Hkv = desc->n_kv_heads;
  p.G = G;
  p.kv_len = desc->kv_len;
  p.L = static_cast<int>(desc->kv_len / parts);
  const float scale = desc->softmax_scale > 0.f
                          ? desc->softmax_scale
                          : static_cast<float>(1.0 / std::sqrt(static_cast<double>(desc->head_dim)));
  p.scale_log2 = scale * cpa::kLog2ed;
  if (parts > 0x7fffffff) return cpa::fail(CP_ATTN_ERR_SHAPE, "decode: too many key runs");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int np = static_cast<int>(parts);
  if (desc->head_dim == 128) {
    st = G <= 4 ? cpa::launch<128, 1>(p, np, s) : G <= 8 ? cpa::launch<128, 2>(p, np, s)
                                                          : cpa::launch<128, 4>(p, np, s);
  } else {
    st = G <= 4 ? cpa::launch<64, 1>(p, np, s) : G <= 8 ? cpa::launch<64, 2>(p, np, s)
                                                         : cpa::launch<64, 4>(p, np, s);
  }
  if (st != CP_ATTN_OK) return st;
  // Pass Q's merge over every rank's (and run's) partial
  return cpa::launch_merge_lse(np, desc->batch, desc->n_q_heads, desc->head_dim, o_part,
                               rows * desc->head_dim, lse_part, rows,
                               static_cast<__nv_bfloat16*>(o), nullptr, lse, s);
}

}  // extern "C"
