// K1: forward ring step on sm_103a (TMA + tcgen05 + TMEM).
//
// One CTA computes one (work item, query head): a 128-row query tile of rank
// q_owner against the run [lo, hi) of non-empty 128-key tiles of rank
// kv_owner ("Built on a fast attention kernel": fully masked blocks are
// skipped; "Ring Attention Algorithms": partial attention of the local
// queries against the visiting KV chunk, merged with the other steps'
// partial results).
//
// Warp roles (192 threads):
//   warps 0-3  softmax + epilogue; thread r owns query row r (TMEM lane r)
//   warp 4     TMA producer (Q once, K/V tiles through a 2-stage ring)
//   warp 5     TMEM owner and single-thread tcgen05.mma issuer
//
// TMEM columns: S double buffer at [0,128) and [128,256), O at [256,256+d).
// The MMA warp issues S(j+1) = Q K_{j+1}^T while the softmax warps turn S(j)
// into P(j); P goes to shared memory in the canonical 128-byte-swizzled
// K-major layout and O += P V_j runs as an SS MMA with V as an MN-major B.
//
// Online softmax in base 2 (scores scaled by scale*log2 e). The running max
// is only raised (and O rescaled in TMEM) when a tile's max exceeds it by
// more than 8, so exponentials stay below 2^8 -- the result is the same
// softmax; only the reference point of the exponentials moves.
//
// S = Q K^T runs on the bf16 inputs (the products are exact in fp32). O += P V
// runs on fp16 operands: P rounded to fp16 keeps 11 significant bits against
// bf16's 8, and V comes from the fp16 copy that step 0 of the ring makes
// (exact for every bf16 value of magnitude in [2^-14, 65504]).
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"

namespace cpa {
namespace {

constexpr int kStages = 2;
constexpr int kThreads = 192;
constexpr float kRescaleThreshold = 8.0f;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

// Barrier slots in shared memory.
enum : int {
  BAR_Q = 0,
  BAR_K = 1,                       // [kStages]
  BAR_V = BAR_K + kStages,         // [kStages]
  BAR_EMPTY = BAR_V + kStages,     // [kStages]
  BAR_S = BAR_EMPTY + kStages,     // [2]
  BAR_P = BAR_S + 2,
  BAR_O = BAR_P + 1,
  BAR_DRAIN = BAR_O + 1,
  BAR_COUNT = BAR_DRAIN + 1
};

template <int D>
struct FwdSmem {
  static constexpr int kTileBytes = 128 * D * 2;  // one Q/K/V tile, bf16
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;
  static constexpr int kV = kK + kStages * kTileBytes;
  static constexpr int kP = kV + kStages * kTileBytes;
  static constexpr int kBar = kP + 128 * 128 * 2;
  static constexpr int kMisc = kBar + BAR_COUNT * 8;
  static constexpr int kBytes = kMisc + 16;
  // 1 KB of slack to align the base; at least 116 KB so that a single CTA
  // (the only one that can hold the 512 TMEM columns) fits per SM.
  static constexpr int kAlloc = (kBytes + 1024) > 118784 ? (kBytes + 1024) : 118784;
};

// Offset of element (row r, column c) of a 128-row bf16 tile stored as
// 64-column blocks of 128 rows x 128 bytes with the 128-byte swizzle (the
// layout TMA writes with CU_TENSOR_MAP_SWIZZLE_128B, and the layout the
// tcgen05 descriptor reads with swizzle mode 128 B).
__device__ __forceinline__ uint32_t sw128_offset(int r, int chunk16) {
  // chunk16: index of the 16-byte chunk along the row (8 bf16 each)
  const int block = chunk16 >> 3;
  const int c = (chunk16 & 7) ^ (r & 7);
  return static_cast<uint32_t>(block * 16384 + r * 128 + (c << 4));
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    step_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using L = FwdSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = ptx::smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_u32 & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_u32 + pad;

  const uint32_t sQ = sbase + L::kQ;
  const uint32_t sK = sbase + L::kK;
  const uint32_t sV = sbase + L::kV;
  const uint32_t sP = sbase + L::kP;
  const uint32_t bar0 = sbase + L::kBar;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int item = blockIdx.x / p.Hq;
  const int h = blockIdx.x % p.Hq;
  const WorkItem w = p.items[item];
  const int kh = h / p.G;
  const int n_tiles = w.hi - w.lo;
  const int64_t q_row0 = static_cast<int64_t>(w.q_owner) * p.n_q + static_cast<int64_t>(w.tile) * 128;
  const int32_t qpos0 = __ldg(p.q_tile_pos + static_cast<int64_t>(w.q_owner) * p.n_qt + w.tile);
  const int64_t kv_row_base = static_cast<int64_t>(w.kv_owner) * p.n_kv;
  const int32_t* kv_tile_pos = p.kv_tile_pos + static_cast<int64_t>(w.kv_owner) * p.n_kt;

  if (threadIdx.x == 0) {
    for (int i = 0; i < BAR_COUNT; ++i) ptx::mbar_init(bar(i), i == BAR_P ? 128u : 1u);
    *s_abort = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 5) {
    ptx::tmem_alloc(ptx::smem_u32(s_tmem), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t tS[2] = {tmem, tmem + 128};
  const uint32_t tO = tmem + 256;

  if (n_tiles > 0 && warp == 4 && lane == 0) {
    // ------------------------------------------------------------ producer
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
    ptx::mbar_arrive_expect_tx(bar(BAR_Q), L::kTileBytes);
    for (int b = 0; b < D / 64; ++b)
      ptx::tma_load_3d(sQ + b * 16384, &tm_q, bar(BAR_Q), b * 64, h, static_cast<int>(q_row0));
    int issued = 0;
    for (int j = 0; j < n_tiles; ++j) {
      const int s = j % kStages;
      if (j >= kStages) {
        if (!ptx::mbar_wait(bar(BAR_EMPTY + s), ((j / kStages) - 1) & 1, s_abort, p.wait_limit_ns)) {
          ptx::record_timeout(p.status, s_abort, 0x100 + j);
          break;
        }
      }
      const int row = static_cast<int>(kv_row_base + static_cast<int64_t>(w.lo + j) * 128);
      ptx::mbar_arrive_expect_tx(bar(BAR_K + s), L::kTileBytes);
      for (int b = 0; b < D / 64; ++b)
        ptx::tma_load_3d(sK + s * L::kTileBytes + b * 16384, &tm_k, bar(BAR_K + s), b * 64, kh, row);
      ptx::mbar_arrive_expect_tx(bar(BAR_V + s), L::kTileBytes);
      for (int b = 0; b < D / 64; ++b)
        ptx::tma_load_3d(sV + s * L::kTileBytes + b * 16384, &tm_v, bar(BAR_V + s), b * 64, kh, row);
      issued = j + 1;
    }
    // Drain: every issued copy must land before the CTA may exit.
    {
      const volatile int never = 0;
      ptx::mbar_wait(bar(BAR_Q), 0, &never, p.wait_limit_ns);
      for (int j = issued > kStages ? issued - kStages : 0; j < issued; ++j) {
        ptx::mbar_wait(bar(BAR_K + j % kStages), (j / kStages) & 1, &never, p.wait_limit_ns);
        ptx::mbar_wait(bar(BAR_V + j % kStages), (j / kStages) & 1, &never, p.wait_limit_ns);
      }
    }
  } else if (n_tiles > 0 && warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop; one elected lane issues each tcgen05
    // instruction, and every wait's outcome is agreed across the warp.
    const uint32_t leader = ptx::elect_one();
    auto wait_w = [&](uint32_t b_, uint32_t parity, int where) -> bool {
      const bool w_ok = ptx::mbar_wait(b_, parity, s_abort, p.wait_limit_ns);
      if (!w_ok && leader) ptx::record_timeout(p.status, s_abort, where);
      return __all_sync(0xffffffffu, w_ok);
    };
    constexpr uint32_t idesc_s = ptx::idesc_bf16(128, 128, 0, 0);
    constexpr uint32_t idesc_o = ptx::idesc_fp16(128, D, 0, 1);  // P and V fp16
    bool ok = wait_w(bar(BAR_Q), 0, 0x200);
    auto issue_pv = [&](int i) -> bool {
      if (!wait_w(bar(BAR_P), i & 1, 0x300 + i)) {
        return false;
      }
      const int s = i % kStages;
      if (!wait_w(bar(BAR_V + s), (i / kStages) & 1, 0x400 + i)) {
        return false;
      }
      ptx::tc_fence_after();
      const uint32_t v_tile = sV + s * L::kTileBytes;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        // A = P [128 q x 128 keys], K-major, swizzled, 64-key blocks of 16 KB
        const uint64_t a = ptx::sdesc_sw128(sP + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
        // B = V [keys x d], d contiguous (MN-major): 8-key groups at 1024 B,
        // 64-column blocks at 16 KB
        const uint64_t b = ptx::sdesc_sw128(v_tile + kk * 2048, 16384, 1024);
        ptx::mma_ss_w(tO, a, b, idesc_o, (i > 0 || kk > 0) ? 1u : 0u, leader);
      }
      ptx::mma_commit_w(bar(BAR_O), leader);
      ptx::mma_commit_w(bar(BAR_EMPTY + s), leader);
      return true;
    };
    for (int j = 0; ok && j < n_tiles; ++j) {
      const int s = j % kStages;
      if (!wait_w(bar(BAR_K + s), (j / kStages) & 1, 0x500 + j)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      const uint32_t k_tile = sK + s * L::kTileBytes;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
        const uint64_t a = ptx::sdesc_sw128(sQ + off, 16, 1024);
        const uint64_t b = ptx::sdesc_sw128(k_tile + off, 16, 1024);
        ptx::mma_ss_w(tS[j & 1], a, b, idesc_s, kk > 0 ? 1u : 0u, leader);
      }
      ptx::mma_commit_w(bar(BAR_S + (j & 1)), leader);
      if (j >= 1 && !issue_pv(j - 1)) {
        ok = false;
        break;
      }
    }
    if (ok) issue_pv(n_tiles - 1);
    // Drain: wait for every MMA this thread issued.
    ptx::mma_commit_w(bar(BAR_DRAIN), leader);
    const volatile int never = 0;
    ptx::mbar_wait(bar(BAR_DRAIN), 0, &never, p.wait_limit_ns);
  } else if (warp < 4) {
    // ------------------------------------------------------------ softmax
    const int r = threadIdx.x;  // query row within the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const int32_t my_pos = qpos0 + r;
    // first visible key of a row: its document start, or the start of its
    // sliding window when that is later
    const int32_t my_ds = ptx::row_lo(p.cu, p.n_cu, p.window, my_pos);
    const int32_t ds_last = ptx::row_lo(p.cu, p.n_cu, p.window, qpos0 + 127);
    float m_used = -INFINITY;  // reference point of the exponentials (base 2)
    float l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int32_t kpos0 = __ldg(kv_tile_pos + w.lo + j);
      const bool full = (kpos0 + 127 <= qpos0) && (kpos0 >= ds_last);
      if (!ptx::mbar_wait(bar(BAR_S + (j & 1)), (j >> 1) & 1, s_abort, p.wait_limit_ns)) {
        ptx::record_timeout(p.status, s_abort, 0x600 + j);
        ok = false;
      }
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      ptx::tc_fence_after();
      float s[128];
#pragma unroll
      for (int c = 0; c < 4; ++c)
        ptx::tmem_ld32(tS[j & 1] + lane_base + c * 32, *reinterpret_cast<float(*)[32]>(s + c * 32));
      if (!full) {
        const int lo = my_ds - kpos0;
        const int hi = my_pos - kpos0;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c < lo || c > hi) s[c] = -INFINITY;
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < 128; ++c) mx = fmaxf(mx, s[c]);
      const float m_tile = mx * p.scale_log2;
      float alpha = 1.f;
      if (m_tile > m_used + kRescaleThreshold) {
        alpha = ptx::ex2(m_used - m_tile);  // 0 when m_used = -inf
        l *= alpha;
        m_used = m_tile;
      }
      const float base = (m_used == -INFINITY) ? 0.f : m_used;
      float rowsum = 0.f;
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        s[c] = ptx::ex2(fmaf(s[c], p.scale_log2, -base));
        rowsum += s[c];
      }
      l += rowsum;
      if (j > 0) {
        // P buffer and O are still in use by PV(j-1)
        if (!ptx::mbar_wait(bar(BAR_O), (j - 1) & 1, s_abort, p.wait_limit_ns)) {
          ptx::record_timeout(p.status, s_abort, 0x700 + j);
          ok = false;
        }
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        ptx::tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            ptx::tmem_ld32(tO + lane_base + c * 32, o);
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] *= alpha;
            ptx::tmem_st32(tO + lane_base + c * 32, o);
          }
        }
      }
      // P (fp16) -> shared memory, swizzled K-major
#pragma unroll
      for (int ch = 0; ch < 16; ++ch) {
        const float* x = s + ch * 8;
        ptx::st_shared_v4(sP + sw128_offset(r, ch), ptx::pack_f16(x[0], x[1]),
                          ptx::pack_f16(x[2], x[3]), ptx::pack_f16(x[4], x[5]),
                          ptx::pack_f16(x[6], x[7]));
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(BAR_P));
    }
    if (ok && n_tiles > 0) {
      if (!ptx::mbar_wait(bar(BAR_O), (n_tiles - 1) & 1, s_abort, p.wait_limit_ns)) {
        ptx::record_timeout(p.status, s_abort, 0x800);
        ok = false;
      }
    }
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      ptx::tc_fence_after();
      // ---------------------------------------------------------- epilogue
      const int64_t g = q_row0 + r;
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const float lse_t = l > 0.f ? (m_used + ptx::lg2(l)) * kLn2 : -INFINITY;
      const int64_t row_off = (g * p.Hq + h) * D;
      const int64_t lse_off = static_cast<int64_t>(h) * p.T_q + g;
      float w_old = 0.f, w_new = 1.f, lse_out = lse_t;
      const bool merge = (p.mode == CP_ATTN_ACCUMULATE) && !p.first;
      float* o_dst = p.o_part;
      float* lse_dst = p.lse_part;
      // WRITE_PARTIAL with bf16 partials: the slot holds bf16 elements
      const bool part_bf16 = p.part_bf16 && p.mode == CP_ATTN_WRITE_PARTIAL;
      __nv_bfloat16* ob = reinterpret_cast<__nv_bfloat16*>(p.o_part);
      if (p.mode == CP_ATTN_WRITE_PARTIAL) {
        const int64_t slot = static_cast<int64_t>(w.kv_owner) * p.T_q * p.Hq * D;
        o_dst += slot;
        ob += slot;
        lse_dst += static_cast<int64_t>(w.kv_owner) * p.Hq * p.T_q;
      }
      if (merge) {
        const float a = lse_dst[lse_off] * kLog2e;
        const float b = lse_t * kLog2e;
        const float M = fmaxf(a, b);
        if (M == -INFINITY) {
          w_old = 0.f;
          w_new = 0.f;
          lse_out = -INFINITY;
        } else {
          const float ea = ptx::ex2(a - M), eb = ptx::ex2(b - M);
          const float sum = ea + eb;
          w_old = ea / sum;
          w_new = eb / sum;
          lse_out = (M + ptx::lg2(sum)) * kLn2;
        }
      }
      lse_dst[lse_off] = lse_out;
      float4* od = reinterpret_cast<float4*>(o_dst + row_off);
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        if (n_tiles > 0) {
          ptx::tmem_ld32(tO + lane_base + c * 32, o);
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = 0.f;
        }
#pragma unroll
        for (int x4 = 0; x4 < 8; ++x4) {
          float4 v;
          v.x = o[x4 * 4 + 0] * inv_l;
          v.y = o[x4 * 4 + 1] * inv_l;
          v.z = o[x4 * 4 + 2] * inv_l;
          v.w = o[x4 * 4 + 3] * inv_l;
          if (merge) {
            const float4 u = od[c * 8 + x4];
            v.x = u.x * w_old + v.x * w_new;
            v.y = u.y * w_old + v.y * w_new;
            v.z = u.z * w_old + v.z * w_new;
            v.w = u.w * w_old + v.w * w_new;
          }
          uint2 pk;
          pk.x = ptx::pack_bf16(v.x, v.y);
          pk.y = ptx::pack_bf16(v.z, v.w);
          if (part_bf16)
            *reinterpret_cast<uint2*>(ob + row_off + c * 32 + x4 * 4) = pk;
          else
            od[c * 8 + x4] = v;
          if (p.o_final) *reinterpret_cast<uint2*>(p.o_final + row_off + c * 32 + x4 * 4) = pk;
        }
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// ===========================================================================
// d = 128: two query heads per CTA in ping-pong.
//
// A CTA takes one query tile and two query heads A and B of the same KV head
// (so both see exactly the same K/V tiles and the same mask). Softmax
// warpgroup A works on S_A(j) while the tensor core runs O_B += P_B V(j-1) and
// S_B(j), and the other way round, so exponentials and MMAs overlap. P is
// written back into its own S columns of TMEM as fp16 pairs (E4M3 quads in
// the F8 instance) and feeds O += P V as the A operand read from tensor
// memory (no shared-memory copy); V is the fp16 copy of the ring.
// K and V stream through separate rings with their own producer warps: a K
// stage is released once both heads' S MMAs have read it, a V stage once both
// O MMAs have, so the next tiles are requested well before they are needed.
// Warps: 0-3 softmax head A, 4-7 softmax head B, 8 Q + K loads, 9 TMEM owner
// + MMA issuer, 10 V loads (352 threads).
// TMEM columns: S_A [0,128) (P_A in [0,64)), S_B [128,256), O_A [256,384),
// O_B [384,512).
constexpr int kThreadsP = 352;
constexpr int kKStagesP = 3;
constexpr int kVStagesP = 2;
// E4M3 tiles are half the size: deeper rings in about two thirds of the space
constexpr int kKStagesF8 = 4;
constexpr int kVStagesF8 = 3;
constexpr int kKStagesMax = 4;
constexpr int kVStagesMax = 3;

enum : int {
  PB_Q = 0,
  PB_K = 1,                      // [kKStagesMax] K tile landed
  PB_V = PB_K + kKStagesMax,     // [kVStagesMax] V tile landed
  PB_KE = PB_V + kVStagesMax,    // [kKStagesMax] K stage free
  PB_VE = PB_KE + kKStagesMax,   // [kVStagesMax] V stage free
  PB_S = PB_VE + kVStagesMax,    // [2] S of head slot ready
  PB_P = PB_S + 2,               // [2 heads][2 halves] P of keys 0-63 / 64-127
                                 // written (128 arrivals)
  PB_O = PB_P + 4,               // [2] final O of head slot ready
  PB_DRAIN = PB_O + 2,
  PB_COUNT = PB_DRAIN + 1
};

// F8: E4M3 operands (one byte per element), else bf16.
template <bool F8>
struct FwdPairSmemT {
  static constexpr int kKS = F8 ? kKStagesF8 : kKStagesP;
  static constexpr int kVS = F8 ? kVStagesF8 : kVStagesP;
  static constexpr int kTile = 128 * 128 * (F8 ? 1 : 2);
  static constexpr int kQ = 0;                          // [2 heads]
  static constexpr int kK = kQ + 2 * kTile;             // [kKS]
  static constexpr int kV = kK + kKS * kTile;           // [kVS]
  static constexpr int kBar = kV + kVS * kTile;
  static constexpr int kMisc = kBar + PB_COUNT * 8;
  static constexpr int kBytes = kMisc + 16;
  // The dynamic shared-memory window starts 1 KB-aligned (checked by the
  // kernel), so no alignment slack is reserved.
  static constexpr int kAlloc = kBytes;
  // The epilogue stages each head's output rows through 32 KB starting at
  // kQ + 32 KB * head: Q and K space, which only the S MMAs read, and those
  // have all completed when a head's last O MMA has.
  static_assert(2 * 32768 <= kV, "epilogue staging must not reach the V ring");
  static_assert(kAlloc > 232448 / 2, "one CTA per SM (each takes all of TMEM)");
};
using FwdPairSmem = FwdPairSmemT<false>;
static_assert(FwdPairSmem::kAlloc <= 232448, "pair kernel shared memory");
static_assert(FwdPairSmemT<true>::kAlloc <= 232448, "pair kernel shared memory");

// F8: Q and K are E4M3 [tokens][heads][d] and tm_v maps V^T, E4M3
// [heads][d][tokens] (keys contiguous, the K-major B operand of O = P V); the
// MMAs are kind::f8f6f4 with K = 32, P goes to TMEM as E4M3 scaled by 2^4
// (probabilities down to 2^-10 of the running maximum stay normal), the
// running maximum moves when it grows by more than 2^4 (so P * 2^4 <= 2^8 =
// 256 < 448, the largest E4M3 value), and the per-tensor descale
// factors p.scales[0..2] (q, k, v) multiply the scores and the output.
// PB: WRITE_PARTIAL with bf16 partials (the slot holds bf16 elements at the
// same element offsets); a separate instance, so that the fp32 epilogue keeps
// its registers.
template <bool F8, bool PB>
__global__ void __launch_bounds__(kThreadsP, 1)
    step_fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const FwdParams p) {
  using L = FwdPairSmemT<F8>;
  constexpr int D = 128;
  constexpr int KS = L::kKS;
  constexpr int VS = L::kVS;
  constexpr int kBoxes = F8 ? 1 : 2;  // 128-byte-wide TMA boxes per 128-row tile
  extern __shared__ __align__(1024) uint8_t smem[];
  const uint32_t sbase = ptx::smem_u32(smem);
  if (sbase & 1023u) {
    // the 128-byte swizzled tiles need a 1 KB-aligned window: report, do nothing
    if (threadIdx.x == 0 &&
        atomicCAS(p.status, 0, static_cast<int>(CP_ATTN_ERR_UNSUPPORTED)) == 0) {
      p.status[1] = static_cast<int>(blockIdx.x);
      p.status[2] = 0x3F00;
    }
    return;
  }
  const uint32_t sQ = sbase + L::kQ;
  const uint32_t sK = sbase + L::kK;
  const uint32_t sV = sbase + L::kV;
  const uint32_t bar0 = sbase + L::kBar;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_pairs = (p.G + 1) >> 1;
  const int Hkv = p.Hq / p.G;
  const int item = blockIdx.x / (Hkv * n_pairs);
  const int rem = blockIdx.x % (Hkv * n_pairs);
  const int kh = rem / n_pairs;
  const int hp = rem % n_pairs;
  const int hA = kh * p.G + 2 * hp;
  const int nh = (p.G - 2 * hp) >= 2 ? 2 : 1;
  const WorkItem w = p.items[item];
  const int n_tiles = w.hi - w.lo;
  const int64_t q_row0 = static_cast<int64_t>(w.q_owner) * p.n_q + static_cast<int64_t>(w.tile) * 128;
  const int32_t qpos0 = __ldg(p.q_tile_pos + static_cast<int64_t>(w.q_owner) * p.n_qt + w.tile);
  const int64_t kv_row_base = static_cast<int64_t>(w.kv_owner) * p.n_kv;
  const int32_t* kv_tile_pos = p.kv_tile_pos + static_cast<int64_t>(w.kv_owner) * p.n_kt;

  if (threadIdx.x == 0) {
    for (int i = 0; i < PB_COUNT; ++i)
      ptx::mbar_init(bar(i), (i >= PB_P && i < PB_P + 4) ? 128u : 1u);
    *s_abort = 0;
    ptx::fence_barrier_init();
  }
  if (warp == 9) {
    ptx::tmem_alloc(ptx::smem_u32(s_tmem), 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *s_tmem;
  // the next ring step may start on SMs this grid leaves idle
  if (threadIdx.x == 0) ptx::grid_dep_launch();

  if (n_tiles > 0 && (warp == 8 || warp == 10) && lane == 0) {
    // ------------------------------------------------------------ producers
    // warp 8: Q once, then K through its ring; warp 10: V through its ring
    const bool is_k = warp == 8;
    const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
    const int NS = is_k ? KS : VS;
    const int full_bar = is_k ? PB_K : PB_V;
    const int free_bar = is_k ? PB_KE : PB_VE;
    const uint32_t ring = is_k ? sK : sV;
    ptx::prefetch_tmap(tm);
    if (is_k) {
      ptx::prefetch_tmap(&tm_q);
      ptx::mbar_arrive_expect_tx(bar(PB_Q), nh * L::kTile);
      for (int hs = 0; hs < nh; ++hs)
        for (int b = 0; b < kBoxes; ++b)
          ptx::tma_load_3d(sQ + hs * L::kTile + b * 16384, &tm_q, bar(PB_Q), b * 64, hA + hs,
                           static_cast<int>(q_row0));
    }
    int issued = 0;
    for (int j = 0; j < n_tiles; ++j) {
      const int s = j % NS;
      if (j >= NS) {
        if (!ptx::mbar_wait(bar(free_bar + s), ((j / NS) - 1) & 1, s_abort, p.wait_limit_ns)) {
          ptx::record_timeout(p.status, s_abort, (is_k ? 0x3100 : 0x3800) + j);
          break;
        }
      }
      const int row = static_cast<int>(kv_row_base + static_cast<int64_t>(w.lo + j) * 128);
      ptx::mbar_arrive_expect_tx(bar(full_bar + s), L::kTile);
      if (F8 && !is_k) {
        // V^T box: 128 keys (bytes) x 128 d rows of head kh
        ptx::tma_load_3d(ring + s * L::kTile, tm, bar(full_bar + s), row, 0, kh);
      } else {
        for (int b = 0; b < kBoxes; ++b)
          ptx::tma_load_3d(ring + s * L::kTile + b * 16384, tm, bar(full_bar + s), b * 64, kh, row);
      }
      issued = j + 1;
    }
    // every issued copy must land before the CTA may exit
    const volatile int never = 0;
    if (is_k) ptx::mbar_wait(bar(PB_Q), 0, &never, p.wait_limit_ns);
    for (int j = issued > NS ? issued - NS : 0; j < issued; ++j)
      ptx::mbar_wait(bar(full_bar + j % NS), (j / NS) & 1, &never, p.wait_limit_ns);
  } else if (n_tiles > 0 && warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop so that descriptors stay warp-uniform;
    // one elected lane issues each tcgen05 instruction.
    const uint32_t leader = ptx::elect_one();
    // kind::f8f6f4 format code 0 is E4M3; kind::f16: S on bf16 Q and K, O on
    // fp16 P and V
    constexpr uint32_t idesc_s = F8 ? ptx::idesc_f16kind(128, 128, 0, 0, 0u)
                                    : ptx::idesc_bf16(128, 128, 0, 0);
    constexpr uint32_t idesc_o = F8 ? ptx::idesc_f16kind(128, D, 0, 0, 0u)
                                    : ptx::idesc_fp16(128, D, 0, 1);
    const uint64_t dQ0 = ptx::sdesc_sw128(sQ, 16, 1024);
    auto wait_set = [&](const auto& bars, const auto& par, int where) -> bool {
      return ptx::wait_phases(bars, par, s_abort, p.wait_limit_ns, p.status, where);
    };
    auto issue_s = [&](int j, int hs) {
      // S = Q K^T: both K-major, two 64-column blocks of 16 KB each
      const uint64_t dk = ptx::sdesc_sw128(sK + (j % KS) * L::kTile, 16, 1024);
      const uint64_t dq = ptx::sdesc_add(dQ0, hs * L::kTile);
      if constexpr (F8) {
        // d = 128 bytes: one swizzle atom, K = 32 elements (32 bytes) per MMA
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          ptx::mma_ss_f8_w(tmem + 128 * hs, ptx::sdesc_add(dq, kk * 32),
                           ptx::sdesc_add(dk, kk * 32), idesc_s, kk > 0 ? 1u : 0u, leader);
      } else {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          ptx::mma_ss_w(tmem + 128 * hs, ptx::sdesc_add(dq, off), ptx::sdesc_add(dk, off), idesc_s,
                        kk > 0 ? 1u : 0u, leader);
        }
      }
      ptx::mma_commit_w(bar(PB_S + hs), leader);
    };
    // O += P V over keys [64 half, 64 half + 64) of tile j
    auto issue_o = [&](int j, int hs, int half) {
      if constexpr (F8) {
        // B = V^T [d][keys] K-major (one swizzle atom); A = P, four E4M3 per
        // column in the head's S columns: 32 keys = 8 columns per MMA
        const uint64_t dv = ptx::sdesc_sw128(sV + (j % VS) * L::kTile, 16, 1024);
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2) {
          const int kk = 2 * half + k2;
          ptx::mma_ts_f8_w(tmem + 256 + 128 * hs, tmem + 128 * hs + kk * 8,
                           ptx::sdesc_add(dv, kk * 32), idesc_o, (j > 0 || kk > 0) ? 1u : 0u,
                           leader);
        }
      } else {
        // B = V [keys][d] MN-major: 8-key groups at 1 KB, d 64..127 at +16 KB
        const uint64_t dv = ptx::sdesc_sw128(sV + (j % VS) * L::kTile, 16384, 1024);
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          // A = P (fp16 pairs in the head's S columns), 16 keys = 8 columns
          const int kk = 4 * half + k4;
          ptx::mma_ts_w(tmem + 256 + 128 * hs, tmem + 128 * hs + kk * 8,
                        ptx::sdesc_add(dv, kk * 2048), idesc_o, (j > 0 || kk > 0) ? 1u : 0u,
                        leader);
        }
      }
    };
    // both halves of O += P V for head slot hs, each once its half of P is
    // written (the first half starts while the second is computed)
    auto issue_o_halves = [&](int jp, int hs, int where) -> bool {
      issue_o(jp, hs, 0);
      const uint32_t b[1] = {bar(PB_P + 2 * hs + 1)};
      const uint32_t ph[1] = {static_cast<uint32_t>(jp & 1)};
      if (!wait_set(b, ph, where)) return false;
      issue_o(jp, hs, 1);
      return true;
    };
    bool ok;
    {
      const uint32_t b[2] = {bar(PB_Q), bar(PB_K)};
      const uint32_t ph[2] = {0u, 0u};
      ok = wait_set(b, ph, 0x3200);
    }
    if (ok) {
      issue_s(0, 0);
      if (nh == 2) issue_s(0, 1);
      ptx::mma_commit_w(bar(PB_KE + 0), leader);
    }
    for (int j = 1; ok && j <= n_tiles; ++j) {
      // head A: O(j-1) then S(j) (S(j) overwrites P(j-1): the pipe is in order)
      const int jp = j - 1;
      const bool more = j < n_tiles;
      {
        // after the last tile there is no K(j): test V(j-1) twice instead
        const uint32_t b[3] = {bar(PB_P + 0), bar(PB_V + jp % VS),
                               more ? bar(PB_K + j % KS) : bar(PB_V + jp % VS)};
        const uint32_t ph[3] = {static_cast<uint32_t>(jp & 1), static_cast<uint32_t>((jp / VS) & 1),
                                more ? static_cast<uint32_t>((j / KS) & 1)
                                     : static_cast<uint32_t>((jp / VS) & 1)};
        if (!wait_set(b, ph, 0x3300 + j)) { ok = false; break; }
      }
      if (!issue_o_halves(jp, 0, 0x3400 + j)) { ok = false; break; }
      if (more) issue_s(j, 0);
      else ptx::mma_commit_w(bar(PB_O + 0), leader);
      if (nh == 2) {
        const uint32_t b[1] = {bar(PB_P + 2)};
        const uint32_t ph[1] = {static_cast<uint32_t>(jp & 1)};
        if (!wait_set(b, ph, 0x3500 + j)) { ok = false; break; }
        if (!issue_o_halves(jp, 1, 0x3900 + j)) { ok = false; break; }
      }
      ptx::mma_commit_w(bar(PB_VE + jp % VS), leader);
      if (nh == 2) {
        if (more) issue_s(j, 1);
        else ptx::mma_commit_w(bar(PB_O + 1), leader);
      }
      if (more) ptx::mma_commit_w(bar(PB_KE + j % KS), leader);
    }
    ptx::mma_commit_w(bar(PB_DRAIN), leader);
    const volatile int never = 0;
    ptx::mbar_wait(bar(PB_DRAIN), 0, &never, p.wait_limit_ns);
    __syncwarp();
  } else if (warp < 8 && (warp >> 2) < nh) {
    // ------------------------------------------------------------ softmax
    const int hs = warp >> 2;
    const int h = hA + hs;
    const int r = threadIdx.x & 127;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + 128 * hs;
    const uint32_t tO = tmem + 256 + 128 * hs;
    const int32_t my_pos = qpos0 + r;
    // first visible key of a row: its document start, or the start of its
    // sliding window when that is later
    const int32_t my_ds = ptx::row_lo(p.cu, p.n_cu, p.window, my_pos);
    const int32_t ds_last = ptx::row_lo(p.cu, p.n_cu, p.window, qpos0 + 127);
    float m_used = -INFINITY;
    float l = 0.f;
    bool ok = true;
    // E4M3 scores carry the q and k descale factors
    const float scale_log2 = F8 ? p.scale_log2 * (__ldg(p.scales) * __ldg(p.scales + 1))
                                : p.scale_log2;
    constexpr float kThreshold = F8 ? 4.f : kRescaleThreshold;
    constexpr float kPExp = F8 ? 4.f : 0.f;  // P is stored as 2^kPExp * p
    int32_t kpos_next = n_tiles > 0 ? __ldg(kv_tile_pos + w.lo) : 0;
    // The epilogue reads this row's fp32 running output back (merge): ask L2
    // for it a few tiles before the end so those reads do not wait on HBM.
    const bool will_merge = p.mode == CP_ATTN_ACCUMULATE && !p.first;
    const int prefetch_at = n_tiles > 3 ? n_tiles - 3 : 0;
    for (int j = 0; j < n_tiles; ++j) {
      const int32_t kpos0 = kpos_next;
      if (j + 1 < n_tiles) kpos_next = __ldg(kv_tile_pos + w.lo + j + 1);
      if (will_merge && j == prefetch_at) {
        const float* row = p.o_part + ((q_row0 + r) * p.Hq + h) * D;
#pragma unroll
        for (int x = 0; x < D * 4 / 128; ++x)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(reinterpret_cast<uint64_t>(row + x * 32)));
      }
      const bool full = (kpos0 + 127 <= qpos0) && (kpos0 >= ds_last);
      if (!ptx::mbar_wait(bar(PB_S + hs), j & 1, s_abort, p.wait_limit_ns)) {
        ptx::record_timeout(p.status, s_abort, 0x3600 + j);
        ok = false;
      }
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      // S(j) complete implies O += P V of tile j-1 complete (issued before it)
      ptx::tc_fence_after();
      float s[128];
      ptx::tmem_ld64x2(tS + lane_base, tS + lane_base + 64, *reinterpret_cast<float(*)[64]>(s),
                       *reinterpret_cast<float(*)[64]>(s + 64));
      if (!full) {
        const int lo = my_ds - kpos0;
        const int hi = my_pos - kpos0;
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c < lo || c > hi) s[c] = -INFINITY;
      }
      // row maximum: eight independent chains of three-input maxima
      float mk[8];
#pragma unroll
      for (int x = 0; x < 8; ++x) mk[x] = ptx::max3(s[2 * x], s[2 * x + 1], s[16 + 2 * x]);
#pragma unroll
      for (int c = 16; c < 128; c += 16) {
#pragma unroll
        for (int x = 0; x < 8; ++x)
          mk[x] = c + 16 < 128 ? ptx::max3(mk[x], s[c + 2 * x + 1], s[c + 16 + 2 * x])
                               : fmaxf(mk[x], s[c + 2 * x + 1]);
      }
      const float mx = fmaxf(ptx::max3(mk[0], mk[1], mk[2]), ptx::max3(mk[3], mk[4], mk[5]));
      const float m_tile = ptx::max3(mx, mk[6], mk[7]) * scale_log2;
      float alpha = 1.f;
      if (m_tile > m_used + kThreshold) {
        alpha = ptx::ex2(m_used - m_tile);
        l *= alpha;
        m_used = m_tile;
      }
      const float base = (m_used == -INFINITY) ? 0.f : m_used;
      const float2 sc2 = make_float2(scale_log2, scale_log2);
      const float2 nb2 = make_float2(kPExp - base, kPExp - base);
      float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                       make_float2(0.f, 0.f)};
      // P of keys 0-63 is handed to the MMA warp before that of keys
      // 64-127. A moved maximum first rescales the running O, which the
      // first half's P V accumulates into (S(j) complete implies O += P V of
      // tile j-1 complete); the rescale runs after the first half's
      // exponentials, when half of the scores are no longer held.
      auto hand_over = [&](int half) {
        if (half == 0 && j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            ptx::tmem_ld32(tO + lane_base + c * 32, o);
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] *= alpha;
            ptx::tmem_st32(tO + lane_base + c * 32, o);
          }
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(PB_P + 2 * hs + half));
      };
      if constexpr (F8) {
        // four keys per column: 64 keys = 16 columns per chunk
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            const int i = c * 64 + 4 * x;
            float2 e0 = ptx::fma2(make_float2(s[i], s[i + 1]), sc2, nb2);
            float2 e1 = ptx::fma2(make_float2(s[i + 2], s[i + 3]), sc2, nb2);
            e0.x = ptx::ex2(e0.x);
            e0.y = ptx::ex2(e0.y);
            e1.x = ptx::ex2(e1.x);
            e1.y = ptx::ex2(e1.y);
            acc[x & 3] = ptx::add2(acc[x & 3], ptx::add2(e0, e1));
            pk[x] = ptx::pack_e4m3x4(e0.x, e0.y, e1.x, e1.y);
          }
          ptx::tmem_st16_nw(tS + lane_base + c * 16, pk);
          hand_over(c);
        }
      } else {
        // P = 2^(s * scale_log2 - base), two columns per instruction, packed
        // to fp16 pairs and stored into this head's S columns [0, 64) chunk
        // by chunk
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            const int i = c * 16 + x;
            float2 e = ptx::fma2(make_float2(s[2 * i], s[2 * i + 1]), sc2, nb2);
            e.x = ptx::ex2(e.x);
            e.y = ptx::ex2(e.y);
            acc[x & 3] = ptx::add2(acc[x & 3], e);
            pk[x] = ptx::pack_f16(e.x, e.y);
          }
          ptx::tmem_st16_nw(tS + lane_base + c * 16, pk);
          if (c & 1) hand_over(c >> 1);
        }
      }
      const float2 acc01 = ptx::add2(acc[0], acc[1]);
      const float2 acc23 = ptx::add2(acc[2], acc[3]);
      const float2 accs = ptx::add2(acc01, acc23);
      l += accs.x + accs.y;
    }
    if (ok && n_tiles > 0) {
      if (!ptx::mbar_wait(bar(PB_O + hs), 0, s_abort, p.wait_limit_ns)) {
        ptx::record_timeout(p.status, s_abort, 0x3700);
        ok = false;
      }
    }
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      // the previous ring step (when this grid was launched chained to it)
      // has finished with the running output and LSE rows read below
      ptx::grid_dep_wait();
      ptx::tc_fence_after();
      const int64_t g = q_row0 + r;
      // l and O carry the 2^kPExp of P; E4M3 V carries its descale factor
      const float inv_l = l > 0.f ? (F8 ? __ldg(p.scales + 2) : 1.f) / l : 0.f;
      const float lse_t = l > 0.f ? (m_used + ptx::lg2(l) - kPExp) * kLn2 : -INFINITY;
      const int64_t lse_off = static_cast<int64_t>(h) * p.T_q + g;
      float w_old = 0.f, w_new = 1.f, lse_out = lse_t;
      const bool merge = (p.mode == CP_ATTN_ACCUMULATE) && !p.first;
      float* o_dst = p.o_part;
      float* lse_dst = p.lse_part;
      __nv_bfloat16* ob = nullptr;  // PB: the bf16 slot
      if (p.mode == CP_ATTN_WRITE_PARTIAL) {
        const int64_t slot = static_cast<int64_t>(w.kv_owner) * p.T_q * p.Hq * D;
        if constexpr (PB) ob = reinterpret_cast<__nv_bfloat16*>(p.o_part) + slot;
        o_dst += slot;
        lse_dst += static_cast<int64_t>(w.kv_owner) * p.Hq * p.T_q;
      }
      if (merge) {
        const float a = lse_dst[lse_off] * kLog2e;
        const float b = lse_t * kLog2e;
        const float M = fmaxf(a, b);
        if (M == -INFINITY) {
          w_old = 0.f;
          w_new = 0.f;
          lse_out = -INFINITY;
        } else {
          const float ea = ptx::ex2(a - M), eb = ptx::ex2(b - M);
          const float sum = ea + eb;
          w_old = ea / sum;
          w_new = eb / sum;
          lse_out = (M + ptx::lg2(sum)) * kLn2;
        }
      }
      // A merge with nothing new (no visible tile) leaves O and LSE as they are.
      const bool keep_old = merge && n_tiles == 0;
      if (!keep_old) lse_dst[lse_off] = lse_out;
      if (!(keep_old && p.o_final == nullptr)) {
        // O rows leave through shared memory so that global accesses are
        // coalesced: per 32-column chunk the warp stages its 32 rows (each
        // thread its own row, 16-byte units XOR-swizzled by row), then
        // writes 4 rows per instruction, 128 contiguous bytes per row.
        // Staging uses this head's Q tile, free once its S MMAs are done.
        ptx::fence_proxy_async_smem();
        uint8_t* stage = smem + L::kQ + hs * 32768 + (warp & 3) * 8192;
        const int sub = lane >> 3;  // row within a group of four
        const int q4 = lane & 7;    // 16-byte unit within the chunk
        const int64_t row_stride = static_cast<int64_t>(p.Hq) * D;
        const int64_t base_off = ((q_row0 + (warp & 3) * 32) * p.Hq + h) * D + q4 * 4;
        // per-row weights of the rows this lane writes: new = a * o + b * old
        const float a_row = inv_l * w_new;
        float a_r[8], b_r[8];
#pragma unroll
        for (int it = 0; it < 8; ++it) {
          a_r[it] = __shfl_sync(0xffffffffu, a_row, it * 4 + sub);
          b_r[it] = __shfl_sync(0xffffffffu, w_old, it * 4 + sub);
        }
        // the running output's rows of chunk c + 1 are requested while chunk
        // c is combined, so the read-backs overlap
        float4 old[8], old_next[8];
        auto load_old = [&](float4 (&dst)[8], int c) {
#pragma unroll
          for (int it = 0; it < 8; ++it)
            dst[it] = *reinterpret_cast<const float4*>(o_dst + base_off + (it * 4 + sub) * row_stride + c * 32);
        };
        if (merge) load_old(old, 0);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          if (n_tiles > 0) {
            ptx::tmem_ld32(tO + lane_base + c * 32, o);
          } else {
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] = 0.f;
          }
          if (merge && c + 1 < D / 32) load_old(old_next, c + 1);
          uint8_t* buf = stage + (c & 1) * 4096;
#pragma unroll
          for (int x4 = 0; x4 < 8; ++x4)
            *reinterpret_cast<float4*>(buf + lane * 128 + ((x4 ^ (lane & 7)) << 4)) =
                make_float4(o[4 * x4], o[4 * x4 + 1], o[4 * x4 + 2], o[4 * x4 + 3]);
          __syncwarp();
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            const int row = it * 4 + sub;
            const float4 t = *reinterpret_cast<const float4*>(buf + row * 128 + ((q4 ^ (row & 7)) << 4));
            float4 v = make_float4(t.x * a_r[it], t.y * a_r[it], t.z * a_r[it], t.w * a_r[it]);
            if (merge) {
              v.x = fmaf(old[it].x, b_r[it], v.x);
              v.y = fmaf(old[it].y, b_r[it], v.y);
              v.z = fmaf(old[it].z, b_r[it], v.z);
              v.w = fmaf(old[it].w, b_r[it], v.w);
            }
            const int64_t off = base_off + row * row_stride + c * 32;
            if constexpr (PB) {
              uint2 pk;
              pk.x = ptx::pack_bf16(v.x, v.y);
              pk.y = ptx::pack_bf16(v.z, v.w);
              *reinterpret_cast<uint2*>(ob + off) = pk;
            } else {
              if (!keep_old) *reinterpret_cast<float4*>(o_dst + off) = v;
              if (p.o_final) {
                uint2 pk;
                pk.x = ptx::pack_bf16(v.x, v.y);
                pk.y = ptx::pack_bf16(v.z, v.w);
                *reinterpret_cast<uint2*>(p.o_final + off) = pk;
              }
            }
          }
          if (merge && c + 1 < D / 32) {
#pragma unroll
            for (int it = 0; it < 8; ++it) old[it] = old_next[it];
          }
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

size_t step_fwd_smem_bytes(int d) {
  return d == 128 ? FwdPairSmem::kAlloc : FwdSmem<64>::kAlloc;
}

int step_fwd_heads_per_cta(int d) { return d == 128 ? 2 : 1; }

cp_attn_status launch_step_fwd(int d, dim3 grid, size_t smem, cudaStream_t s,
                               const CUtensorMap& tq, const CUtensorMap& tk,
                               const CUtensorMap& tv, const FwdParams& p, bool chained) {
  static bool attr_done[3] = {false, false, false};
  cudaError_t err;
  if (d == 128) {
    const bool pb = p.part_bf16 != 0;
    auto kernel = pb ? step_fwd_pair_kernel<false, true> : step_fwd_pair_kernel<false, false>;
    if (!attr_done[pb ? 2 : 1]) {
      err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
      if (err != cudaSuccess) return fail(CP_ATTN_ERR_CUDA, std::string("step_fwd attr: ") + cudaGetErrorString(err));
      attr_done[pb ? 2 : 1] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreadsP);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = chained ? 1 : 0;
    err = cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, p);
    if (err != cudaSuccess) return fail(CP_ATTN_ERR_CUDA, std::string("step_fwd launch: ") + cudaGetErrorString(err));
  } else {
    if (!attr_done[0]) {
      err = cudaFuncSetAttribute(step_fwd_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
      if (err != cudaSuccess) return fail(CP_ATTN_ERR_CUDA, std::string("step_fwd attr: ") + cudaGetErrorString(err));
      attr_done[0] = true;
    }
    step_fwd_kernel<64><<<grid, kThreads, smem, s>>>(tq, tk, tv, p);
  }
  err = cudaGetLastError();
  if (err != cudaSuccess) return fail(CP_ATTN_ERR_CUDA, std::string("step_fwd launch: ") + cudaGetErrorString(err));
  count_launch();
  return CP_ATTN_OK;
}

size_t step_fwd_fp8_smem_bytes() { return FwdPairSmemT<true>::kAlloc; }

cp_attn_status launch_step_fwd_fp8(dim3 grid, size_t smem, cudaStream_t s,
                                   const CUtensorMap& tq, const CUtensorMap& tk,
                                   const CUtensorMap& tvt, const FwdParams& p, bool chained) {
  static bool attr_done[2] = {false, false};
  cudaError_t err;
  const bool pb = p.part_bf16 != 0;
  auto kernel = pb ? step_fwd_pair_kernel<true, true> : step_fwd_pair_kernel<true, false>;
  if (!attr_done[pb ? 1 : 0]) {
    err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
    if (err != cudaSuccess) return fail(CP_ATTN_ERR_CUDA, std::string("step_fwd_fp8 attr: ") + cudaGetErrorString(err));
    attr_done[pb ? 1 : 0] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreadsP);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = chained ? 1 : 0;
  err = cudaLaunchKernelEx(&cfg, kernel, tq, tk, tvt, p);
  if (err != cudaSuccess) return fail(CP_ATTN_ERR_CUDA, std::string("step_fwd_fp8 launch: ") + cudaGetErrorString(err));
  count_launch();
  return CP_ATTN_OK;
}

}  // namespace cpa
