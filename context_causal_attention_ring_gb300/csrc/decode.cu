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
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>

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
  extern __shared__ __align__(1024) uint8_t smem[];
  float* q_s = reinterpret_cast<float*>(smem + S::kQ);
  float* s_s = reinterpret_cast<float*>(smem + S::kS);
  float* o_s = reinterpret_cast<float*>(smem + S::kO);
  float* st_max = reinterpret_cast<float*>(smem + S::kStat);
  float* st_sum = st_max + kDecMaxG;
  const uint32_t kv_s = ptx::smem_u32(smem + S::kKV);
  // the merge that follows waits for this grid to complete (see decode_tc_kernel)
  if (threadIdx.x == 0) ptx::grid_dep_launch();

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

// K9: the same partial attention on the tensor cores (head_dim 128, runs of
// 128, 256 or 512 keys: an item is one run of one KV head of one sequence).
// The G <= 16 query heads of a KV head form the N = 16 side of two products
// per 128-key tile, both accumulated in TMEM:
//   S^T  = K Q^T    (M = 128 keys, N = 16 heads, K = d)
//   O^T += V^T P^T  (M = d, N = 16 heads, K = keys)
// The grid is persistent (as many CTAs as the SMs hold, a multiple of Hkv);
// each CTA keeps one KV head and takes that head's items one after another
// from a work counter. The K tiles and then the V tiles of its items stream
// through a TMA ring (two 32 KB slots for bf16, four 16 KB slots for E4M3,
// six at 16 heads), so the next item's tiles load while the current one is
// in its softmax; the producer starts the first slots' loads before the
// block's setup barrier. An item's scores fit in TMEM (16 columns per tile),
// so the softmax is one pass between the two products: per head, the maximum
// and the sum over the run, reduced across the four warps that hold its keys
// through shared memory. P goes to shared memory as the B operand of O^T.
// The CTA merges the partial results of its consecutive items of one
// sequence in TMEM and writes one partial per such run. Query rows past G
// are zero; only the group's heads, rounded up to 4, 8 or 16, go through the
// softmax.
// Warps: SW softmax and epilogue warps (4, or 8 for 16 heads: warp w holds
// keys / columns of d 32 (w mod 4) .. +31 and a quarter or half of the
// heads), then the TMA producer and the TMEM owner and MMA issuer. About
// 75 KB (E4M3), 107 KB (E4M3, 16 heads) or 87 KB (bf16) of shared memory:
// two CTAs share an SM, three for E4M3 when the group has at most eight
// heads.
constexpr int kTcN = 16;                    // MMA N: the query heads, padded
constexpr int kTcMaxTiles = kDecMaxL / 128;

constexpr int kDecMaxSlots = 6;  // ring slots, at most (see dec_slots)

enum : int {
  TB_FULL = 0,                      // [kDecMaxSlots] tile of the slot landed
  TB_EMPTY = kDecMaxSlots,          // [kDecMaxSlots] slot read by its MMAs
  TB_S = 2 * kDecMaxSlots,          // all scores of the run in TMEM
  TB_P = 2 * kDecMaxSlots + 1,      // [4] softmax-warp arrivals: P of tile t in shared memory
  TB_O = 2 * kDecMaxSlots + 5,      // O^T complete
  TB_RED = 2 * kDecMaxSlots + 6,    // softmax-warp arrivals per phase: partial maxima, then sums
  TB_Q = 2 * kDecMaxSlots + 7,      // softmax-warp arrivals: the next group's query rows written
  TB_DONE = 2 * kDecMaxSlots + 8,   // every MMA of the CTA complete
  TB_OST = 2 * kDecMaxSlots + 9,    // softmax-warp arrivals: a run's O staged for its store
  TB_SFREE = 2 * kDecMaxSlots + 10, // the staging buffer's last store has read it (once)
  TB_ITEM = 2 * kDecMaxSlots + 11,  // [kDecItemRing] the producer published an item
  TB_COUNT = 2 * kDecMaxSlots + 11 + 8
};
constexpr int kDecItemRing = 8;  // items published ahead of their consumers, at most

// Ring slots of the tensor-core decode: bf16 tiles (32 KB) two; E4M3 tiles
// (16 KB) four, six at 16 heads (two CTAs per SM either way), so that the
// next item's first K tiles load while the current item's V tiles wait for
// P.
constexpr int dec_slots(bool f8, int nh) { return f8 ? (nh == 16 ? 6 : 4) : 2; }

// F8: E4M3 K rows and V^T tiles (one byte per element, 16 KB per tile), the
// query rows and P in E4M3; else bf16 (32 KB tiles).
template <bool F8, int SLOTS = dec_slots(F8, 4)>
struct DecTcSmem {
  static constexpr int kElt = F8 ? 1 : 2;
  static constexpr int kSlots = SLOTS;
  static_assert(SLOTS <= kDecMaxSlots, "one full and one empty barrier per slot");
  static constexpr int kTile = 128 * 128 * kElt;            // a K or V tile
  static constexpr int kRing = 0;                           // [kSlots]
  static constexpr int kQ = kRing + kSlots * kTile;         // [16][128] query rows
  static constexpr int kP = kQ + kTcN * 128 * kElt;         // [16][512] P
  static constexpr int kRed = kP + kTcN * kDecMaxL * kElt;  // [max | sum][4 warps][16] f32
  static constexpr int kQs = kRed + 2 * 4 * kTcN * 4;       // [16] f32 query scales (F8)
  static constexpr int kBar = kQs + kTcN * 4;
  static constexpr int kMisc = kBar + (TB_COUNT + 4) * 8;  // TMEM address, abort flag
  static constexpr int kItem = kMisc + 16;                   // [kDecItemRing] int item ring
  static constexpr int kBytes = kItem + kDecItemRing * 4;
};
// three E4M3 CTAs of the four-slot ring share an SM (1 KB reserved per CTA)
static_assert(3 * (DecTcSmem<true, 4>::kBytes + 1024) <= 233472, "three CTAs per SM");

struct DecTcParams {
  const __nv_bfloat16* q;  // [B][Hq][128]
  float* o_part;           // [parts][B][Hq][128]
  float* lse_part;         // [parts][Hq][B]
  int B, Hq, Hkv, G;
  int64_t kv_len;
  int L;                   // keys per part: 128, 256 or 512
  int parts;               // parts per sequence: kv_len / L
  int* counters;           // [Hkv] work counters, zero at launch
  float scale_log2;
  int32_t* status;         // [4] device status word
  uint64_t wait_limit_ns;
  const float* kv_scales;  // F8: device [2] descale factors of K and V
};

// Byte offset of element (row, col) of a K-major 8-bit operand with 16 rows:
// 128-column blocks of 16 x 128 bytes (2 KB), 16-byte units XOR-swizzled by
// row.
__device__ __forceinline__ uint32_t kmaj16_off8(int row, int col) {
  const int chunk = ((col & 127) >> 4) ^ (row & 7);
  return static_cast<uint32_t>((col >> 7) * 2048 + row * 128 + (chunk << 4) + (col & 15));
}

// Byte offset of element (row, col) of a K-major bf16 operand with 16 rows:
// 64-column blocks of 16 x 128 bytes (2 KB), 16-byte units XOR-swizzled by
// row (the 128-byte swizzle).
__device__ __forceinline__ uint32_t kmaj16_off(int row, int col) {
  const int chunk = ((col & 63) >> 3) ^ (row & 7);
  return static_cast<uint32_t>((col >> 6) * 2048 + row * 128 + (chunk << 4) + ((col & 7) << 1));
}

// Tile i of a run of nt K tiles and then nt V tiles (rows row0 + 128 (i mod
// nt) of KV head kh) into ring slot `slot`, completing on that slot's full
// barrier.
template <bool F8>
__device__ __forceinline__ void dec_issue_tile(const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                               uint32_t ring, uint32_t bar0, int slot, int i,
                                               int nt, int row0, int kh) {
  using S = DecTcSmem<F8>;
  const uint32_t full = bar0 + 8u * static_cast<uint32_t>(TB_FULL + slot);
  const int row = row0 + (i % nt) * 128;
  ptx::mbar_arrive_expect_tx(full, S::kTile);
  if (F8 && i >= nt) {
    // V^T box: 128 keys (bytes) x 128 d rows of head kh
    ptx::tma_load_3d(ring + slot * S::kTile, tm_v, full, row, 0, kh);
  } else {
#pragma unroll
    for (int blk = 0; blk < (F8 ? 1 : 2); ++blk)
      ptx::tma_load_3d(ring + slot * S::kTile + blk * 16384, i < nt ? tm_k : tm_v, full, blk * 64,
                       kh, row);
  }
}

// F8: tm_k maps E4M3 K [B*kv_len][Hkv][128] (128-byte boxes), tm_v maps V^T
// E4M3 [Hkv][128][B*kv_len]; each head's query row is quantized here with its
// own scale, S^T and O^T are kind::f8f6f4 with K = 32, and P goes to shared
// memory as E4M3 scaled by 2^8 (P <= 1 against the run's exact maximum).
// The warp-wide reduction (max or sum) of each of a lane's N values (N = 4 or
// 8, one per head), by halving: at each of the first log2 N steps a lane
// keeps half of its values, sends the other half to its partner and combines
// the halves it holds, so that the last steps work on a single value. It
// costs N - 1 + 5 - log2 N shuffles instead of 5 N. Lane l returns the
// reduction of value l >> (5 - log2 N).
template <int N, bool MAX>
__device__ __forceinline__ float warp_reduce_heads(const float (&v)[N], int lane) {
  static_assert(N == 4 || N == 8, "four or eight values per lane");
  auto op = [](float a, float b) { return MAX ? fmaxf(a, b) : a + b; };
  float w[N];
#pragma unroll
  for (int k = 0; k < N; ++k) w[k] = v[k];
#pragma unroll
  for (int n = N, off = 16; n > 1; n >>= 1, off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int k = 0; k < n / 2; ++k) {
      const float keep = upper ? w[k + n / 2] : w[k];
      const float send = upper ? w[k] : w[k + n / 2];
      w[k] = op(keep, __shfl_xor_sync(0xffffffffu, send, off));
    }
  }
  constexpr int kDone = N == 8 ? 3 : 2;  // offsets 16 .. 32 >> kDone used above
#pragma unroll
  for (int off = 16 >> kDone; off > 0; off >>= 1) w[0] = op(w[0], __shfl_xor_sync(0xffffffffu, w[0], off));
  return w[0];
}

// Softmax warps of the tensor-core decode: eight (two groups of four, eight
// heads each) when all 16 columns of N are heads, else four.
constexpr int dec_softmax_warps(int nh) { return nh == 16 ? 8 : 4; }
// CTAs per SM the kernel is compiled for: three fit in shared memory; with
// eight softmax warps the registers allow two.
constexpr int dec_min_ctas(int nh) { return nh == 16 ? 2 : 3; }

// NH: the group's query heads rounded up to 4, 8 or 16 (a compile-time
// count, so that the per-head softmax chains interleave without branches);
// columns past NH are padding of N and are never read.
template <bool F8, int NH>
__global__ void __launch_bounds__(32 * (dec_softmax_warps(NH) + 2), dec_min_ctas(NH))
    decode_tc_kernel(
    const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
    const DecTcParams p) {
  using S = DecTcSmem<F8, dec_slots(F8, NH)>;
  constexpr int NSL = S::kSlots;
  constexpr int SW = dec_softmax_warps(NH);  // softmax warps; then the producer, the MMA warp
  constexpr int HPW = NH * 4 / SW;           // heads per softmax warp
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = ptx::smem_u32(smem);
  if (sbase & 1023u) {
    // the 128-byte swizzled tiles need a 1 KB-aligned window: report, do nothing
    if (threadIdx.x == 0 &&
        atomicCAS(p.status, 0, static_cast<int>(CP_ATTN_ERR_UNSUPPORTED)) == 0) {
      p.status[1] = static_cast<int>(blockIdx.x);
      p.status[2] = 0x9F00;
    }
    return;
  }
  // the merge that follows may be scheduled once every CTA has started; it
  // waits for this grid to complete before it reads the partials
  if (threadIdx.x == 0) ptx::grid_dep_launch();
  const uint32_t sRing = sbase + S::kRing;
  const uint32_t sQ = sbase + S::kQ;
  const uint32_t sP = sbase + S::kP;
  float* red = reinterpret_cast<float*>(smem + S::kRed);
  const uint32_t bar0 = sbase + S::kBar;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + S::kMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + S::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.G;
  const int nt = p.L / 128;
  // The items are (sequence b, part, KV head kh), numbered kh fastest. The
  // grid is a multiple of Hkv and CTA c keeps KV head kh = c mod Hkv: its
  // first item is the (c / Hkv)-th (b, part) of that head and each further
  // one is taken from the head's work counter as the CTA gets to it, so CTAs
  // that run faster take more items. A CTA's items thus come in increasing
  // (b, part) order: its query rows change only with the sequence, and the
  // heads advance together, so the CTAs running at one time read every KV
  // head of the same rows (adjacent in memory). The producer publishes each
  // item (its number, or -1 once there are none) in a ring of kDecItemRing
  // entries with one barrier each; the other warps read it there. Fewer than
  // 2^31 items: batch * kv_len < 2^31 and Hkv <= 128.
  int* s_item = reinterpret_cast<int*>(smem + S::kItem);
  struct Item {
    int part, kh, b, row0;
  };
  auto item_of = [&](int i) {
    Item r;
    r.kh = i % p.Hkv;
    const int bp = i / p.Hkv;
    r.b = bp / p.parts;
    r.part = bp - r.b * p.parts;
    r.row0 = static_cast<int>(static_cast<int64_t>(r.b) * p.kv_len +
                              static_cast<int64_t>(r.part) * p.L);
    return r;
  };
  // the producer's j-th item (j > 0 takes a counter ticket), or -1
  auto take_item = [&](int j) -> int {
    const int kh = static_cast<int>(blockIdx.x) % p.Hkv;
    const int per_head = static_cast<int>(gridDim.x) / p.Hkv;
    const int bp = j == 0 ? static_cast<int>(blockIdx.x) / p.Hkv
                          : per_head + atomicAdd(p.counters + kh, 1);
    return bp < p.B * p.parts ? bp * p.Hkv + kh : -1;
  };
  const int item0 = take_item(0);  // no ticket: every thread knows it
  const Item first = item_of(item0 < 0 ? 0 : item0);

  // tiles of the first item that need no free slot; tile i of the CTA's
  // item j is the (j * 2 nt + i)-th tile through the ring
  const int n_first = item0 >= 0 ? (2 * nt < NSL ? 2 * nt : NSL) : 0;
  if (warp == SW && lane == 0) {
    // the producer sets up the barriers itself, publishes the first item and
    // starts the first ring of loads at once, so that they overlap the query
    // rows and the TMEM allocation; nobody else touches a barrier before the
    // block barrier
    for (int i = 0; i < TB_COUNT; ++i)
      ptx::mbar_init(bar(i), ((i >= TB_P && i < TB_P + kTcMaxTiles) || i == TB_RED || i == TB_Q ||
                              i == TB_OST)
                                 ? 32u * SW
                                 : 1u);
    *s_abort = 0;
    ptx::fence_barrier_init();
    s_item[0] = item0;
    ptx::mbar_arrive(bar(TB_ITEM));
    for (int i = 0; i < n_first; ++i)
      dec_issue_tile<F8>(&tm_k, &tm_v, sRing, bar0, i, i, nt, first.row0, first.kh);
  }
  if (warp == SW + 1) {
    ptx::tmem_alloc(ptx::smem_u32(s_tmem), 128);
    ptx::tmem_relinquish();
  }
  // E4M3 descale factors of K and V, loaded before they are needed
  float kv_sk = 1.f, kv_sv = 1.f;
  if (F8 && warp < SW) {
    kv_sk = __ldg(p.kv_scales);
    kv_sv = __ldg(p.kv_scales + 1);
  }
  // the query rows of group (b, kh) as the B operand of S^T, written by the
  // softmax warps
  auto write_q = [&](int b, int kh) {
    if constexpr (F8) {
      // each head's query row to E4M3 with its own scale (amax / 448); warp w
      // takes rows w, w + SW, ...: lane l holds d = 4l .. 4l + 3
      float* qs = reinterpret_cast<float*>(smem + S::kQs);
      // all of the warp's rows' loads first, so that their latencies overlap
      uint2 u[kTcN / SW];
#pragma unroll
      for (int j = 0; j < kTcN / SW; ++j) {
        const int h = warp + SW * j;
        u[j] = make_uint2(0u, 0u);
        if (h < G)
          u[j] = __ldg(reinterpret_cast<const uint2*>(
              p.q + (static_cast<int64_t>(b) * p.Hq + kh * G + h) * 128 + 4 * lane));
      }
#pragma unroll
      for (int j = 0; j < kTcN / SW; ++j) {
        const int h = warp + SW * j;
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[j].x));
        const float2 c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[j].y));
        const float x[4] = {a.x, a.y, c.x, c.y};
        float m = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float inv = m > 0.f ? 448.f / m : 1.f;
        if (lane == 0) qs[h] = m > 0.f ? m / 448.f : 1.f;
        const uint32_t q4 = ptx::pack_e4m3x4(x[0] * inv, x[1] * inv, x[2] * inv, x[3] * inv);
        *reinterpret_cast<uint32_t*>(smem + S::kQ + kmaj16_off8(h, 4 * lane)) = q4;
      }
    } else {
      // K-major rows; rows past G zero
      uint4 v[kTcN * 16 / (32 * SW)];
#pragma unroll
      for (int j = 0; j < kTcN * 16 / (32 * SW); ++j) {
        const int c = threadIdx.x + 32 * SW * j;
        const int h = c >> 4;
        v[j] = make_uint4(0u, 0u, 0u, 0u);
        if (h < G)
          v[j] = __ldg(reinterpret_cast<const uint4*>(
              p.q + (static_cast<int64_t>(b) * p.Hq + kh * G + h) * 128 + (c & 15) * 8));
      }
#pragma unroll
      for (int j = 0; j < kTcN * 16 / (32 * SW); ++j) {
        const int c = threadIdx.x + 32 * SW * j;
        *reinterpret_cast<uint4*>(smem + S::kQ + kmaj16_off(c >> 4, (c & 15) * 8)) = v[j];
      }
    }
    ptx::fence_proxy_async_smem();
  };
  if (warp < SW && item0 >= 0) write_q(first.b, first.kh);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  volatile int* v_item = s_item;
  const volatile int never = 0;

  if (warp == SW && lane == 0) {
    // ------------------------------------------------------------ producer
    int issued = n_first;  // ring tiles issued so far
    bool ok = true;
    int idx = item0;
    for (int j = 0; ok && idx >= 0; ++j) {
      const Item c = item_of(idx);
      // the next item is taken once this one's first tile is on its way, so
      // that the counter's round trip overlaps the waits for free slots
      int next = -1;
      bool taken = false;
      for (int i = j == 0 ? n_first : 0; i < 2 * nt; ++i) {
        const int g = j * 2 * nt + i;
        const int slot = g % NSL;
        if (g >= NSL &&
            !ptx::mbar_wait(bar(TB_EMPTY + slot), ((g / NSL) - 1) & 1, s_abort, p.wait_limit_ns)) {
          ptx::record_timeout(p.status, s_abort, 0x9100 + i);
          ok = false;
          break;
        }
        dec_issue_tile<F8>(&tm_k, &tm_v, sRing, bar0, slot, i, nt, c.row0, c.kh);
        issued = g + 1;
        if (!taken) {
          next = take_item(j + 1);
          taken = true;
        }
      }
      if (!ok) break;
      if (!taken) next = take_item(j + 1);
      // publish item j + 1 (its entry's previous reader, item j + 1 - 8, is
      // done: the producer runs at most a ring of tiles ahead of the MMAs)
      v_item[(j + 1) % kDecItemRing] = next;
      ptx::mbar_arrive(bar(TB_ITEM + (j + 1) % kDecItemRing));
      idx = next;
    }
    // every issued copy must land before the CTA may exit
    for (int g = issued > NSL ? issued - NSL : 0; g < issued; ++g)
      ptx::mbar_wait(bar(TB_FULL + (g % NSL)), (g / NSL) & 1, &never, p.wait_limit_ns);
  } else if (warp == SW + 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t leader = ptx::elect_one();
    auto wait_w = [&](uint32_t b_, uint32_t parity, int where) -> bool {
      const bool w_ok = ptx::mbar_wait(b_, parity, s_abort, p.wait_limit_ns);
      if (!w_ok && leader) ptx::record_timeout(p.status, s_abort, where);
      return __all_sync(0xffffffffu, w_ok);
    };
    // bf16: K-major A and B for S^T, MN-major A (V) for O^T. E4M3 (format 0
    // of kind::f8f6f4): K-major everywhere (V arrives as V^T)
    constexpr uint32_t idesc_s = F8 ? ptx::idesc_f16kind(128, kTcN, 0, 0, 0u)
                                    : ptx::idesc_bf16(128, kTcN, 0, 0);
    constexpr uint32_t idesc_o = F8 ? ptx::idesc_f16kind(128, kTcN, 0, 0, 0u)
                                    : ptx::idesc_bf16(128, kTcN, 1, 0);
    const uint64_t dQ = ptx::sdesc_sw128(sQ, 16, 1024);
    const uint64_t dP = ptx::sdesc_sw128(sP, 16, 1024);
    bool ok = true;
    int n_q = 0;  // query-row rewrites waited for
    Item prev = first;
    int run_b = -1;  // the sequence of the run the O^T accumulator holds
    for (int j = 0; ok; ++j) {
      int idx = item0;
      if (j > 0) {
        if (!wait_w(bar(TB_ITEM + j % kDecItemRing), (j / kDecItemRing) & 1, 0x9C00)) {
          ok = false;
          break;
        }
        idx = v_item[j % kDecItemRing];
      }
      if (idx < 0) break;
      const Item c = item_of(idx);
      const bool new_q = c.b != prev.b || c.kh != prev.kh;
      prev = c;
      // a new run starts the O^T accumulator afresh (the softmax warps read
      // the previous run out before they hand over this item's P)
      const uint32_t acc0 = c.b != run_b ? 0u : 1u;
      run_b = c.b;
      if (new_q) {
        // the softmax warps wrote the new group's query rows
        if (!wait_w(bar(TB_Q), n_q & 1, 0x9A00)) { ok = false; break; }
        ++n_q;
        ptx::tc_fence_after();
      }
      for (int t = 0; ok && t < nt; ++t) {
        const int g = j * 2 * nt + t;
        const int slot = g % NSL;
        if (!wait_w(bar(TB_FULL + slot), (g / NSL) & 1, 0x9200 + t)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint64_t dK = ptx::sdesc_sw128(sRing + slot * S::kTile, 16, 1024);
        if constexpr (F8) {
          // K tile [128 keys][128 d bytes]: one swizzle atom, 32 d per MMA
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            ptx::mma_ss_f8_w(tmem + kTcN * t, ptx::sdesc_add(dK, kk * 32),
                             ptx::sdesc_add(dQ, kk * 32), idesc_s, kk > 0 ? 1u : 0u, leader);
        } else {
          // K tile [128 keys][128 d] in two 64-column blocks of 16 KB
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            ptx::mma_ss_w(tmem + kTcN * t, ptx::sdesc_add(dK, (kk >> 2) * 16384 + (kk & 3) * 32),
                          ptx::sdesc_add(dQ, (kk >> 2) * 2048 + (kk & 3) * 32), idesc_s,
                          kk > 0 ? 1u : 0u, leader);
        }
        ptx::mma_commit_w(bar(TB_EMPTY + slot), leader);
      }
      if (!ok) break;
      ptx::mma_commit_w(bar(TB_S), leader);
      // O^T += V^T P^T tile by tile, each as soon as its P and its V are in
      // (an early tile's product frees its V slot for the next item's K)
      for (int t = 0; ok && t < nt; ++t) {
        const int g = j * 2 * nt + nt + t;
        const int slot = g % NSL;
        if (!wait_w(bar(TB_P + t), j & 1, 0x9300 + t)) { ok = false; break; }
        if (!wait_w(bar(TB_FULL + slot), (g / NSL) & 1, 0x9400 + t)) { ok = false; break; }
        ptx::tc_fence_after();
        if constexpr (F8) {
          // V^T tile [128 d][128 keys bytes] as the K-major A; P as the
          // K-major B, 128 keys per 2 KB block, 32 keys per MMA
          const uint64_t dV = ptx::sdesc_sw128(sRing + slot * S::kTile, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            ptx::mma_ss_f8_w(tmem + 64, ptx::sdesc_add(dV, kk * 32),
                             ptx::sdesc_add(dP, t * 2048 + kk * 32), idesc_o,
                             (t > 0 || kk > 0) ? 1u : acc0, leader);
        } else {
          // V tile as the MN-major A of O^T (M = d: d 64..127 at +16 KB; K =
          // keys, 16 keys = 2 KB per step); P as the K-major B, 64 keys per
          // 2 KB block
          const uint64_t dV = ptx::sdesc_sw128(sRing + slot * S::kTile, 16384, 1024);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            ptx::mma_ss_w(tmem + 64, ptx::sdesc_add(dV, kk * 2048),
                          ptx::sdesc_add(dP, (2 * t + (kk >> 2)) * 2048 + (kk & 3) * 32),
                          idesc_o, (t > 0 || kk > 0) ? 1u : acc0, leader);
        }
        ptx::mma_commit_w(bar(TB_EMPTY + slot), leader);
      }
      if (!ok) break;
      ptx::mma_commit_w(bar(TB_O), leader);
    }
    // every MMA issued above must complete before the TMEM is released
    ptx::mma_commit_w(bar(TB_DONE), leader);
    ptx::mbar_wait(bar(TB_DONE), 0, &never, p.wait_limit_ns);
    __syncwarp();
  } else if (warp < SW) {
    // ------------------------------------------------------------ softmax
    // warp w: TMEM lanes 32 (w mod 4) .. +31 (key of each tile, then column
    // of d) and heads [h0, h0 + HPW)
    const int t = threadIdx.x & 127;
    const int qw = warp & 3;
    const int h0 = (warp >> 2) * HPW;
    const uint32_t lane_base = static_cast<uint32_t>(qw * 32) << 16;
    constexpr int kHeadShift = HPW == 8 ? 2 : 3;  // warp_reduce_heads: lane l ends with head l >> kHeadShift
    // base-2 score factor per head (E4M3: times the query row's and K's
    // descale factors)
    const float* qs = reinterpret_cast<const float*>(smem + S::kQs);
    // E4M3: O^T carries 2^8 of P and V's descale factor
    const float oscale = F8 ? kv_sv * (1.f / 256.f) : 1.f;
    // The CTA merges its consecutive items of one sequence (a run) as it
    // goes, in the online form of the log-sum-exp merge ("Ring Attention
    // Algorithms"): the run's maximum m and sum l per head live in TMEM
    // columns kRunM and kRunL (one copy per lane), its O in the O^T
    // accumulator, which the items' O^T = V^T P^T products keep adding into.
    // P is taken against m, raised to an item's maximum when that is larger
    // (O and l are then scaled by 2^(m_old - m_new) before the item's O^T
    // products), so P <= 1 as within an item. A run leaves as one partial in
    // the slot of its first part; its other parts' slots get LSE = -inf
    // (weight 0 in the merge that follows). The O rows of the group's G
    // heads are contiguous in o_part: they are staged [head][d] in the P
    // buffer (the last O^T products have read P) and leave in one bulk store.
    constexpr uint32_t kRunM = 96, kRunL = 112;
    int run_b = -1, run_part = 0, n_flush = 0;
    auto flush = [&](int kh) -> bool {
      uint32_t o[HPW], m[HPW], l_[HPW];
      ptx::tmem_ld_n<HPW>(tmem + lane_base + 64 + h0, o);
      ptx::tmem_ld_n<HPW>(tmem + lane_base + kRunM + h0, m);
      ptx::tmem_ld_n<HPW>(tmem + lane_base + kRunL + h0, l_);
      float* stage = reinterpret_cast<float*>(smem + S::kP);
#pragma unroll
      for (int h = 0; h < HPW; ++h) {
        const int hh = h0 + h;
        if (hh < G) {
          const float lh = __uint_as_float(l_[h]);
          stage[hh * 128 + t] = __uint_as_float(o[h]) * (__frcp_rn(lh) * oscale);
          if (t == hh)
            p.lse_part[(static_cast<int64_t>(run_part) * p.Hq + kh * G + hh) * p.B + run_b] =
                (__uint_as_float(m[h]) + ptx::lg2(lh)) * kLn2d;
        }
      }
      ptx::fence_proxy_async_smem();
      ptx::mbar_arrive(bar(TB_OST));
      bool f_ok = true;
      if (threadIdx.x == 0) {
        f_ok = ptx::mbar_wait(bar(TB_OST), n_flush & 1, s_abort, p.wait_limit_ns);
        if (f_ok) {
          const int64_t obase = (static_cast<int64_t>(run_part) * p.B + run_b) * p.Hq + kh * G;
          ptx::bulk_store(p.o_part + obase * 128, sP, static_cast<uint32_t>(G) * 512u);
          ptx::bulk_commit();
        } else {
          ptx::record_timeout(p.status, s_abort, 0x9E00);
        }
      }
      ++n_flush;
      return f_ok;
    };
    bool ok = true;
    int n_q = 0;
    int last_j = -1;  // the last item this CTA's softmax warps finished
    Item prev = first;
    for (int j = 0; ok; ++j) {
      int idx = item0;
      if (j > 0) {
        ok = ptx::mbar_wait(bar(TB_ITEM + j % kDecItemRing), (j / kDecItemRing) & 1, s_abort,
                            p.wait_limit_ns);
        if (!ok) ptx::record_timeout(p.status, s_abort, 0x9D00);
        if (!__all_sync(0xffffffffu, ok)) break;
        idx = v_item[j % kDecItemRing];
      }
      if (idx < 0) break;
      const Item c = item_of(idx);
      const bool new_q = c.b != prev.b || c.kh != prev.kh;
      prev = c;
      if (new_q) {
        // the previous item's S^T products are complete (its softmax waited
        // for them), so the query rows may be rewritten
        write_q(c.b, c.kh);
        ptx::mbar_arrive(bar(TB_Q));
        // all softmax warps' rows (and E4M3 scales) written
        ok = ptx::mbar_wait(bar(TB_Q), n_q & 1, s_abort, p.wait_limit_ns);
        if (!ok) ptx::record_timeout(p.status, s_abort, 0x9B00);
        ++n_q;
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      // S^T of this item complete implies the previous item's O^T products
      // complete (issued before it)
      ok = ptx::mbar_wait(bar(TB_S), j & 1, s_abort, p.wait_limit_ns);
      if (!ok) ptx::record_timeout(p.status, s_abort, 0x9500);
      if (!__all_sync(0xffffffffu, ok)) break;
      ptx::tc_fence_after();
      const bool run_start = c.b != run_b;
      if (run_start && run_b >= 0) {
        // the previous run leaves before this item's O^T products start anew
        ok = flush(c.kh);
        if (!__all_sync(0xffffffffu, ok)) break;
      }
      float x[kTcMaxTiles][HPW];
      float M[HPW], l[HPW];
      {
        float sf[HPW];
#pragma unroll
        for (int h = 0; h < HPW; ++h) sf[h] = p.scale_log2;
        if constexpr (F8) {
#pragma unroll
          for (int h = 0; h < HPW; ++h) sf[h] *= qs[h0 + h] * kv_sk;
        }
#pragma unroll
        for (int i = 0; i < kTcMaxTiles; ++i) {
          if (i < nt) {
            uint32_t r[HPW];
            ptx::tmem_ld_n<HPW>(tmem + lane_base + kTcN * i + h0, r);
#pragma unroll
            for (int h = 0; h < HPW; ++h) x[i][h] = __uint_as_float(r[h]) * sf[h];
          } else {
#pragma unroll
            for (int h = 0; h < HPW; ++h) x[i][h] = -INFINITY;
          }
        }
        // per head: maximum over the thread's keys, the warp, then the four
        // warps of the head's group. Columns past NH are skipped here and
        // below: their P is left as it is and only feeds O^T columns that
        // are never read.
#pragma unroll
        for (int h = 0; h < HPW; ++h) {
          float m = x[0][h];
#pragma unroll
          for (int i = 1; i < kTcMaxTiles; ++i) m = fmaxf(m, x[i][h]);
          M[h] = m;
        }
        const float m = warp_reduce_heads<HPW, true>(M, lane);
        if ((lane & ((1 << kHeadShift) - 1)) == 0) red[qw * kTcN + h0 + (lane >> kHeadShift)] = m;
      }
      // P is written after this phase, over the previous run's O staging:
      // its store must have read it
      if (threadIdx.x == 0) ptx::bulk_wait_read();
      ptx::mbar_arrive(bar(TB_RED));
      ok = ptx::mbar_wait(bar(TB_RED), 0, s_abort, p.wait_limit_ns);
      if (!ok) ptx::record_timeout(p.status, s_abort, 0x9600);
      if (!__all_sync(0xffffffffu, ok)) break;
      // the run's reference maximum per head: the item's at a run's start,
      // else raised to it (O and l scaled down) when it is larger
      uint32_t rm[HPW], rl[HPW];
      if (run_start) {
#pragma unroll
        for (int h = 0; h < HPW; ++h) {
          const int hh = h0 + h;
          rm[h] = __float_as_uint(
              fmaxf(fmaxf(red[hh], red[kTcN + hh]), fmaxf(red[2 * kTcN + hh], red[3 * kTcN + hh])));
          rl[h] = __float_as_uint(0.f);
        }
      } else {
        ptx::tmem_ld_n<HPW>(tmem + lane_base + kRunM + h0, rm);
        ptx::tmem_ld_n<HPW>(tmem + lane_base + kRunL + h0, rl);
        float fac[HPW];
        bool moved = false;
#pragma unroll
        for (int h = 0; h < HPW; ++h) {
          const int hh = h0 + h;
          const float mi =
              fmaxf(fmaxf(red[hh], red[kTcN + hh]), fmaxf(red[2 * kTcN + hh], red[3 * kTcN + hh]));
          const float mr = __uint_as_float(rm[h]);
          fac[h] = 1.f;
          if (mi > mr) {
            fac[h] = ptx::ex2(mr - mi);
            rm[h] = __float_as_uint(mi);
            rl[h] = __float_as_uint(__uint_as_float(rl[h]) * fac[h]);
            moved = true;
          }
        }
        if (__any_sync(0xffffffffu, moved)) {
          // O^T: TMEM lane = column t of d, column h = query head
          uint32_t o[HPW];
          ptx::tmem_ld_n<HPW>(tmem + lane_base + 64 + h0, o);
#pragma unroll
          for (int h = 0; h < HPW; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * fac[h]);
          ptx::tmem_st_n<HPW>(tmem + lane_base + 64 + h0, o);
        }
      }
      // P = 2^(x - m) (bf16 or E4M3 into shared memory) tile by tile, each
      // tile handed to the MMA warp as soon as it is written (the first
      // hand-over also covers the O^T scaling above), and the per-head sums
      float mr[HPW];
#pragma unroll
      for (int h = 0; h < HPW; ++h) {
        mr[h] = __uint_as_float(rm[h]);
        l[h] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < kTcMaxTiles; ++i) {
        if (i < nt) {
#pragma unroll
          for (int h = 0; h < HPW; ++h) {
            const float e = ptx::ex2(x[i][h] - mr[h]);
            l[h] += e;
            if constexpr (F8) {
              // 2^8 P <= 256: probabilities down to 2^-14 stay normal
              smem[S::kP + kmaj16_off8(h0 + h, i * 128 + t)] =
                  static_cast<uint8_t>(ptx::pack_e4m3x4(e * 256.f, 0.f, 0.f, 0.f) & 0xFFu);
            } else {
              *reinterpret_cast<__nv_bfloat16*>(smem + S::kP + kmaj16_off(h0 + h, i * 128 + t)) =
                  __float2bfloat16_rn(e);
            }
          }
          ptx::fence_proxy_async_smem();
          // this warp's reads of S^T and its scaling of O^T are done
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar(TB_P + i));
        }
      }
      {
        const float sm = warp_reduce_heads<HPW, false>(l, lane);
        if ((lane & ((1 << kHeadShift) - 1)) == 0)
          red[4 * kTcN + qw * kTcN + h0 + (lane >> kHeadShift)] = sm;
      }
      ptx::mbar_arrive(bar(TB_RED));
      ok = ptx::mbar_wait(bar(TB_RED), 1, s_abort, p.wait_limit_ns);
      if (!ok) ptx::record_timeout(p.status, s_abort, 0x9700);
      if (!__all_sync(0xffffffffu, ok)) break;
      {
        const float* rs = red + 4 * kTcN;
#pragma unroll
        for (int h = 0; h < HPW; ++h) {
          const int hh = h0 + h;
          rl[h] = __float_as_uint(__uint_as_float(rl[h]) +
                                  ((rs[hh] + rs[kTcN + hh]) + (rs[2 * kTcN + hh] + rs[3 * kTcN + hh])));
          // a part inside a run carries no partial of its own
          if (!run_start && hh < G && t == hh)
            p.lse_part[(static_cast<int64_t>(c.part) * p.Hq + c.kh * G + hh) * p.B + c.b] =
                -INFINITY;
        }
      }
      ptx::tmem_st_n<HPW>(tmem + lane_base + kRunM + h0, rm);
      ptx::tmem_st_n<HPW>(tmem + lane_base + kRunL + h0, rl);
      if (run_start) {
        run_b = c.b;
        run_part = c.part;
      }
      last_j = j;
    }
    // the last item's O^T products complete before the last run leaves
    if (ok && last_j >= 0) {
      ok = ptx::mbar_wait(bar(TB_O), last_j & 1, s_abort, p.wait_limit_ns);
      if (!ok) ptx::record_timeout(p.status, s_abort, 0x9800);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) ptx::tc_fence_after();
    }
    // The last run leaves. Its staging may follow another run's in the same
    // item (no P was written in between, so nothing has waited for that
    // store to read the buffer): thread 0 waits for it and lets the others
    // go on.
    if (ok && run_b >= 0) {
      if (threadIdx.x == 0) {
        ptx::bulk_wait_read();
        ptx::mbar_arrive(bar(TB_SFREE));
      }
      ok = ptx::mbar_wait(bar(TB_SFREE), 0, s_abort, p.wait_limit_ns);
      if (!ok) ptx::record_timeout(p.status, s_abort, 0x9F10);
      if (__all_sync(0xffffffffu, ok)) flush(prev.kh);
    }
    if (threadIdx.x == 0) ptx::bulk_wait_all();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == SW + 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 128);
  }
}

// Raises a kernel's dynamic shared-memory limit in the current context. A
// function attribute belongs to the context, so it is set on every call (a
// cheap driver call) rather than remembered.
cp_attn_status set_smem_limit(const void* fn, size_t bytes, const char* what) {
  const cudaError_t err =
      cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (err != cudaSuccess) {
    cudaGetLastError();
    return fail(CP_ATTN_ERR_CUDA, std::string(what) + " attr: " + cudaGetErrorString(err));
  }
  return CP_ATTN_OK;
}

// CTAs of kernel `fn` (one of kResidentSlots instances, `slot`) that the
// current device holds at once, from the kernel's registers, its shared
// memory and its threads against the SM's limits. It depends only on the
// device and the kernel, so it is kept per (device, slot).
constexpr int kResidentSlots = 6;
constexpr int kResidentDevices = 64;
cp_attn_status resident_ctas(const void* fn, int slot, int threads, size_t smem, int* out) {
  static std::atomic<int> cache[kResidentDevices][kResidentSlots];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess && dev >= 0 && dev < kResidentDevices) {
    const int v = cache[dev][slot].load(std::memory_order_relaxed);
    if (v > 0) {
      *out = v;
      return CP_ATTN_OK;
    }
  }
  int sms = 0, regs_sm = 0, smem_sm = 0, smem_rsv = 0, thr_sm = 0, blk_sm = 0;
  cudaFuncAttributes fa{};
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&smem_rsv, cudaDevAttrReservedSharedMemoryPerBlock, dev);
  if (e == cudaSuccess)
    e = cudaDeviceGetAttribute(&thr_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&blk_sm, cudaDevAttrMaxBlocksPerMultiprocessor, dev);
  if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, fn);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(CP_ATTN_ERR_CUDA, std::string("decode occupancy: ") + cudaGetErrorString(e));
  }
  // registers are given out per warp in units of 256
  const int warp_regs = ((fa.numRegs * 32 + 255) / 256) * 256;
  const int by_regs = regs_sm / (warp_regs * ((threads + 31) / 32));
  const int by_smem =
      smem_sm / static_cast<int>(smem + fa.sharedSizeBytes + static_cast<size_t>(smem_rsv));
  int per_sm = by_regs < by_smem ? by_regs : by_smem;
  if (thr_sm / threads < per_sm) per_sm = thr_sm / threads;
  if (blk_sm < per_sm) per_sm = blk_sm;
  if (sms * per_sm <= 0) return fail(CP_ATTN_ERR_CUDA, "decode occupancy: no CTA fits on an SM");
  *out = sms * per_sm;
  if (dev >= 0 && dev < kResidentDevices) cache[dev][slot].store(*out, std::memory_order_relaxed);
  return CP_ATTN_OK;
}

// Keys per CTA. head_dim 128 (the tensor-core kernel, two CTAs per SM): the
// largest of 512, 256, 128 that divides the shard and still leaves about two
// CTAs per SM, else 128 if it divides the shard. Otherwise (and for
// head_dim 64, four CTAs per SM): the largest of 512, 256, 128, 64 that
// leaves about four CTAs per SM; 64 if none does.
int pick_part_len(int64_t shard, int64_t ctas_per_part, int head_dim) {
  if (head_dim == 128) {
    for (int L : {kDecMaxL, 256, 128})
      if (shard % L == 0 && (shard / L) * ctas_per_part >= 152 * 2) return L;
    if (shard % 128 == 0) return 128;
  }
  for (int L : {kDecMaxL, 256, 128})
    if (shard % L == 0 && (shard / L) * ctas_per_part >= 152 * 4) return L;
  return kDecTile;
}

// Device status word of the tensor-core decode kernel (its bounded waits
// record a timeout there), one per device. Its device address is looked up in
// the current context on every call (the lookup allocates nothing): an address
// kept from an earlier call could belong to a context that has since been
// destroyed.
__device__ int32_t g_decode_status[4];

cp_attn_status decode_status_address(int32_t** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return fail(CP_ATTN_ERR_CUDA, "decode: no current CUDA device");
  }
  void* ptr = nullptr;
  const cudaError_t err = cudaGetSymbolAddress(&ptr, g_decode_status);
  if (err != cudaSuccess || ptr == nullptr) {
    cudaGetLastError();
    return fail(CP_ATTN_ERR_CUDA, std::string("decode: status word lookup failed: ") +
                                      cudaGetErrorString(err));
  }
  *out = static_cast<int32_t*>(ptr);
  return CP_ATTN_OK;
}

// F8: k is E4M3 [B*kv_len][Hkv][128], v the E4M3 V^T [Hkv][128][B*kv_len].
template <bool F8>
cp_attn_status launch_tc(const void* k, const void* v, const DecTcParams& p, int parts,
                         cudaStream_t s) {
  CUtensorMap tk, tv;
  const int64_t rows = static_cast<int64_t>(p.B) * p.kv_len;
  cp_attn_status st = F8 ? encode_u8_map(&tk, k, rows, p.Hkv, 128, false)
                         : encode_bf16_rows_map(&tk, k, rows, p.Hkv, 128);
  if (st != CP_ATTN_OK) return st;
  if ((st = F8 ? encode_u8_map(&tv, v, rows, p.Hkv, 128, true)
               : encode_bf16_rows_map(&tv, v, rows, p.Hkv, 128)) != CP_ATTN_OK)
    return st;
  const int nh = p.G <= 4 ? 4 : p.G <= 8 ? 8 : 16;
  const size_t smem = nh == 16 ? DecTcSmem<F8, dec_slots(F8, 16)>::kBytes
                               : DecTcSmem<F8, dec_slots(F8, 4)>::kBytes;
  auto kernel = nh == 4 ? decode_tc_kernel<F8, 4>
                : nh == 8 ? decode_tc_kernel<F8, 8> : decode_tc_kernel<F8, 16>;
  const int ai = nh == 4 ? 0 : nh == 8 ? 1 : 2;
  const int threads = 32 * (dec_softmax_warps(nh) + 2);
  int resident = 0;
  cp_attn_status st2 = set_smem_limit(reinterpret_cast<const void*>(kernel), smem, "decode_tc");
  if (st2 == CP_ATTN_OK) {
    // all of the unified L1 / shared memory as shared memory, so that the
    // occupancy below counts the CTAs that really fit
    const cudaError_t e = cudaFuncSetAttribute(reinterpret_cast<const void*>(kernel),
                                               cudaFuncAttributePreferredSharedMemoryCarveout,
                                               static_cast<int>(cudaSharedmemCarveoutMaxShared));
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(CP_ATTN_ERR_CUDA, std::string("decode_tc carveout: ") + cudaGetErrorString(e));
    }
    st2 = resident_ctas(reinterpret_cast<const void*>(kernel), F8 * 3 + ai, threads, smem, &resident);
  }
  if (st2 != CP_ATTN_OK) return st2;
  // A persistent grid: as many CTAs as fit on the device at once, rounded
  // down to a multiple of Hkv (at least Hkv: with more KV heads than resident
  // CTAs the rest wait for a slot), and no more than there are items. Its
  // CTAs take their items from the per-KV-head work counters, zeroed here on
  // the stream. items = B * parts * Hkv is a multiple of Hkv too.
  if (p.counters == nullptr) return fail(CP_ATTN_ERR_INVALID_ARG, "decode_tc: no work counters");
  DecTcParams q = p;
  q.parts = parts;
  const int64_t items = static_cast<int64_t>(p.B) * p.Hkv * parts;
  int64_t grid_n = resident - resident % p.Hkv;
  if (grid_n < p.Hkv) grid_n = p.Hkv;
  if (grid_n > items) grid_n = items;
  {
    const cudaError_t e = cudaMemsetAsync(q.counters, 0, sizeof(int) * p.Hkv, s);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(CP_ATTN_ERR_CUDA, std::string("decode_tc counters: ") + cudaGetErrorString(e));
    }
  }
  const unsigned grid = static_cast<unsigned>(grid_n);
  kernel<<<grid, threads, smem, s>>>(tk, tv, q);
  const cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return fail(CP_ATTN_ERR_CUDA, std::string("decode_tc: ") + cudaGetErrorString(err));
  count_launch();
  return CP_ATTN_OK;
}

// Workspace of a decode call: the fp32 partial outputs [parts][B][Hq][d], the
// partial LSEs [parts][Hq][B] and the tensor-core kernel's work counters
// [Hkv], each at a 256-byte offset.
struct DecodeLayout {
  size_t lse_off, ctr_off, total;
};
int64_t n_parts(const cp_attn_decode_desc* d);
DecodeLayout decode_layout(const cp_attn_decode_desc* d) {
  const int64_t parts = n_parts(d);
  const int64_t rows = static_cast<int64_t>(d->batch) * d->n_q_heads;
  auto up = [](size_t x) { return ((x + 255) / 256) * 256; };
  DecodeLayout l;
  l.lse_off = up(static_cast<size_t>(parts * rows * d->head_dim) * 4);
  l.ctr_off = up(l.lse_off + static_cast<size_t>(parts * rows) * 4);
  l.total = l.ctr_off + static_cast<size_t>(d->n_kv_heads) * 4;
  return l;
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
  const int L = pick_part_len(shard, static_cast<int64_t>(d->cp) * d->n_kv_heads * d->batch,
                             d->head_dim);
  return d->kv_len / L;
}

template <int D, int HPG>
cp_attn_status launch(const DecParams& p, int parts, cudaStream_t s) {
  const size_t smem = DecSmem<D>::kBytes;
  const cp_attn_status st =
      set_smem_limit(reinterpret_cast<const void*>(decode_partial_kernel<D, HPG>), smem, "decode");
  if (st != CP_ATTN_OK) return st;
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
  *bytes = cpa::decode_layout(desc).total;
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
  const cpa::DecodeLayout lay = cpa::decode_layout(desc);
  float* o_part = static_cast<float*>(workspace);
  float* lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + lay.lse_off);
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
  if (desc->head_dim == 128 && p.L % 128 == 0 &&
      static_cast<int64_t>(desc->batch) * desc->kv_len <= 0x7fffffff) {
    cpa::DecTcParams tp;
    tp.q = p.q;
    tp.o_part = p.o_part;
    tp.lse_part = p.lse_part;
    tp.B = p.B;
    tp.Hq = p.Hq;
    tp.Hkv = p.Hkv;
    tp.G = p.G;
    tp.kv_len = p.kv_len;
    tp.L = p.L;
    tp.scale_log2 = p.scale_log2;
    tp.wait_limit_ns = 1000000000ull;
    if ((st = cpa::decode_status_address(&tp.status)) != CP_ATTN_OK) return st;
    tp.kv_scales = nullptr;
    tp.counters = reinterpret_cast<int*>(static_cast<char*>(workspace) + lay.ctr_off);
    st = cpa::launch_tc<false>(k, v, tp, np, s);
  } else if (desc->head_dim == 128) {
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
                               static_cast<__nv_bfloat16*>(o), nullptr, lse, s, false,
                               /*pdl=*/true);
}

cp_attn_status cp_attn_decode_fp8(const cp_attn_decode_desc* desc, const void* q, const void* k8,
                                  const void* vt8, const float* kv_scales, void* o, float* lse,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  cpa::clear_error();
  size_t need = 0;
  cp_attn_status st = cp_attn_decode_workspace_size(desc, &need);
  if (st != CP_ATTN_OK) return st;
  if (desc->head_dim != 128)
    return cpa::fail(CP_ATTN_ERR_UNSUPPORTED, "decode_fp8: head_dim must be 128");
  if (!q || !k8 || !vt8 || !kv_scales || !o || !lse || !workspace)
    return cpa::fail(CP_ATTN_ERR_INVALID_ARG, "decode_fp8: null pointer");
  for (const void* ptr : {q, k8, vt8, static_cast<const void*>(kv_scales),
                          static_cast<const void*>(o), static_cast<const void*>(lse),
                          static_cast<const void*>(workspace)})
    if (reinterpret_cast<uintptr_t>(ptr) % 16)
      return cpa::fail(CP_ATTN_ERR_INVALID_ARG, "decode_fp8: pointers must be 16-byte aligned");
  if (workspace_bytes < need) return cpa::fail(CP_ATTN_ERR_SHAPE, "decode_fp8: workspace too small");
  const int64_t parts = cpa::n_parts(desc);
  const int L = static_cast<int>(desc->kv_len / parts);
  if (L % 128 || static_cast<int64_t>(desc->batch) * desc->kv_len > 0x7fffffff)
    return cpa::fail(CP_ATTN_ERR_SHAPE,
                     "decode_fp8: kv_len / cp must be a multiple of 128 and batch * kv_len < 2^31");
  const int G = desc->n_q_heads / desc->n_kv_heads;
  const int64_t rows = static_cast<int64_t>(desc->batch) * desc->n_q_heads;
  const cpa::DecodeLayout lay = cpa::decode_layout(desc);
  cpa::DecTcParams tp;
  tp.q = static_cast<const __nv_bfloat16*>(q);
  tp.o_part = static_cast<float*>(workspace);
  tp.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + lay.lse_off);
  tp.counters = reinterpret_cast<int*>(static_cast<char*>(workspace) + lay.ctr_off);
  tp.B = desc->batch;
  tp.Hq = desc->n_q_heads;
  tp.Hkv = desc->n_kv_heads;
  tp.G = G;
  tp.kv_len = desc->kv_len;
  tp.L = L;
  const float scale = desc->softmax_scale > 0.f
                          ? desc->softmax_scale
                          : static_cast<float>(1.0 / std::sqrt(static_cast<double>(desc->head_dim)));
  tp.scale_log2 = scale * cpa::kLog2ed;
  tp.wait_limit_ns = 1000000000ull;
  tp.kv_scales = kv_scales;
  if ((st = cpa::decode_status_address(&tp.status)) != CP_ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int np = static_cast<int>(parts);
  if ((st = cpa::launch_tc<true>(k8, vt8, tp, np, s)) != CP_ATTN_OK) return st;
  return cpa::launch_merge_lse(np, desc->batch, desc->n_q_heads, desc->head_dim, tp.o_part,
                               rows * desc->head_dim, tp.lse_part, rows,
                               static_cast<__nv_bfloat16*>(o), nullptr, lse, s, false,
                               /*pdl=*/true);
}

cp_attn_status cp_attn_decode_sync_status(void* stream) {
  cpa::clear_error();
  int32_t* status = nullptr;
  cp_attn_status st = cpa::decode_status_address(&status);
  if (st != CP_ATTN_OK) return st;
  cudaError_t err = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess)
    return cpa::fail(CP_ATTN_ERR_CUDA, std::string("decode_sync_status: ") + cudaGetErrorString(err));
  int32_t h[4] = {0, 0, 0, 0};
  err = cudaMemcpy(h, status, sizeof(h), cudaMemcpyDeviceToHost);
  if (err == cudaSuccess && h[0] != 0) err = cudaMemset(status, 0, sizeof(h));
  if (err != cudaSuccess)
    return cpa::fail(CP_ATTN_ERR_CUDA, std::string("decode_sync_status: ") + cudaGetErrorString(err));
  if (h[0] != 0)
    return cpa::fail(static_cast<cp_attn_status>(h[0]),
                     "decode: device-side error in block " + std::to_string(h[1]) +
                         " at wait site 0x" + [&] {
                           char b[16];
                           std::snprintf(b, sizeof(b), "%x", h[2]);
                           return std::string(b);
                         }());
  return CP_ATTN_OK;
}

}  // extern "C"
