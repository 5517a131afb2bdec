// K2: backward ring step on sm_103a (TMA + tcgen05 + TMEM).
//
// One CTA owns one 128-key tile of rank kv_owner and one KV head, and loops
// over the G query heads of that KV head times the run [lo, hi) of visible
// query tiles of rank q_owner. With the merged (global) LSE and
// delta = rowsum(dO * O) of each query row, every iteration computes
//   S^T  = K Q^T                     (keys x queries, TMEM)
//   dP^T = V dO^T                    (TMEM)
//   P^T  = exp(scale S^T - LSE)      masked, -> fp16 in shared memory
//   dS^T = P^T (dP^T - delta)        -> fp16 in shared memory
//   dV  += P^T dO,  dK += dS^T Q     (TMEM accumulators for the whole CTA)
//   dQ   = dS K                      (TMEM, then fp32 atomics into dq)
// so dK and dV are summed over the GQA group inside the CTA and written once
// per step. The backward pass is called once per ring step like the forward
// ("Built on a fast attention kernel": P2P runs the kernel per ring step in
// the forward and backward pass).
//
// Warp roles (192 threads): warps 0-3 compute (thread j owns key row j for
// P/dS and query row j for the dQ read-out), warp 4 TMA producer, warp 5
// TMEM owner and tcgen05.mma issuer.
// TMEM columns: S^T [0,128), dP^T and then dQ [128,256), dV [256,256+d),
// dK [256+d,256+2d).
// All operands are fp16 (exact copies of the bf16 inputs, and P / dS rounded
// to fp16): the probabilities keep 11 significant bits instead of 8, which
// keeps the fp32 gradients within 1e-2 of the exact ones.
#include <cmath>

#include "kernels.h"
#include "ptx.cuh"

namespace cpa {
namespace {

constexpr int kThreads = 192;
constexpr float kLog2e = 1.44269504088896340736f;

enum : int {
  BAR_KV = 0,
  BAR_QF = 1,  // [2] Q and dO of a stage landed
  BAR_QE = 3,  // [2] stage free again
  BAR_S = 5,
  BAR_DP = 6,
  BAR_P = 7,       // 128 arrivals: P^T and dS^T written
  BAR_DQ = 8,      // all MMAs of the iteration done
  BAR_DQFREE = 9,  // 128 arrivals: dQ read out of TMEM
  BAR_DRAIN = 10,
  BAR_ROW = 11,    // 128 arrivals: this iteration's LSE/delta row staged
  BAR_COUNT = 12
};

template <int D>
struct BwdSmem {
  static constexpr int kStages = D == 128 ? 1 : 2;
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kQ = kV + kTileBytes;                 // [kStages]
  static constexpr int kDO = kQ + kStages * kTileBytes;      // [kStages]
  static constexpr int kPt = kDO + kStages * kTileBytes;     // P^T  [128 keys x 128 q] bf16
  static constexpr int kDSt = kPt + 128 * 128 * 2;           // dS^T [128 keys x 128 q] bf16
  static constexpr int kRow = kDSt + 128 * 128 * 2;          // lse2/delta [2][2][128] f32
  static constexpr int kBar = kRow + 2 * 2 * 128 * 4;
  static constexpr int kMisc = kBar + BAR_COUNT * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = (kBytes + 1024) > 118784 ? (kBytes + 1024) : 118784;
};

__device__ __forceinline__ uint32_t sw128_offset(int r, int chunk16) {
  const int block = chunk16 >> 3;
  const int c = (chunk16 & 7) ^ (r & 7);
  return static_cast<uint32_t>(block * 16384 + r * 128 + (c << 4));
}

// End (exclusive) of the document that contains `pos`: the smallest
// cu[i] > pos.
__device__ __forceinline__ int32_t doc_end(const int32_t* __restrict__ cu, int n_cu,
                                           int32_t pos) {
  int lo = 0, hi = n_cu - 1;  // cu[lo] <= pos < cu[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(cu + mid) <= pos) lo = mid;
    else hi = mid;
  }
  return __ldg(cu + hi);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    step_bwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_do, const BwdParams p) {
  using L = BwdSmem<D>;
  constexpr int NS = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = ptx::smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_u32 & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_u32 + pad;
  const uint32_t sK = sbase + L::kK;
  const uint32_t sV = sbase + L::kV;
  const uint32_t sQ = sbase + L::kQ;
  const uint32_t sDO = sbase + L::kDO;
  const uint32_t sPt = sbase + L::kPt;
  const uint32_t sDSt = sbase + L::kDSt;
  float* s_row = reinterpret_cast<float*>(smem + L::kRow);  // [buf][0=lse2,1=delta][128]
  const uint32_t bar0 = sbase + L::kBar;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int item = blockIdx.x / p.Hkv;
  const int kh = blockIdx.x % p.Hkv;
  const WorkItem w = p.items[item];
  const int n_qtiles = w.hi - w.lo;
  const int n_iter = n_qtiles * p.G;
  const int64_t kv_row0 = static_cast<int64_t>(w.kv_owner) * p.n_kv + static_cast<int64_t>(w.tile) * 128;
  const int32_t kpos0 = __ldg(p.kv_tile_pos + static_cast<int64_t>(w.kv_owner) * p.n_kt + w.tile);
  const int32_t* q_tile_pos = p.q_tile_pos + static_cast<int64_t>(w.q_owner) * p.n_qt;
  const int64_t q_row_base = static_cast<int64_t>(w.q_owner) * p.n_q;

  if (threadIdx.x == 0) {
    for (int i = 0; i < BAR_COUNT; ++i)
      ptx::mbar_init(bar(i), (i == BAR_P || i == BAR_DQFREE || i == BAR_ROW) ? 128u : 1u);
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
  const uint32_t tS = tmem;
  const uint32_t tDP = tmem + 128;  // dP^T, then dQ
  const uint32_t tDV = tmem + 256;
  const uint32_t tDK = tmem + 256 + D;

  if (n_iter > 0 && warp == 4 && lane == 0) {
    // ------------------------------------------------------------ producer
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
    ptx::prefetch_tmap(&tm_do);
    ptx::mbar_arrive_expect_tx(bar(BAR_KV), 2 * L::kTileBytes);
    for (int b = 0; b < D / 64; ++b) {
      ptx::tma_load_3d(sK + b * 16384, &tm_k, bar(BAR_KV), b * 64, kh, static_cast<int>(kv_row0));
      ptx::tma_load_3d(sV + b * 16384, &tm_v, bar(BAR_KV), b * 64, kh, static_cast<int>(kv_row0));
    }
    int issued = 0;
    for (int it = 0; it < n_iter; ++it) {
      const int s = it % NS;
      if (it >= NS) {
        if (!ptx::mbar_wait(bar(BAR_QE + s), ((it / NS) - 1) & 1, s_abort, p.wait_limit_ns)) {
          ptx::record_timeout(p.status, s_abort, 0x1100 + it);
          break;
        }
      }
      const int h = kh * p.G + it / n_qtiles;
      const int row = static_cast<int>(q_row_base + static_cast<int64_t>(w.lo + it % n_qtiles) * 128);
      ptx::mbar_arrive_expect_tx(bar(BAR_QF + s), 2 * L::kTileBytes);
      for (int b = 0; b < D / 64; ++b) {
        ptx::tma_load_3d(sQ + s * L::kTileBytes + b * 16384, &tm_q, bar(BAR_QF + s), b * 64, h, row);
        ptx::tma_load_3d(sDO + s * L::kTileBytes + b * 16384, &tm_do, bar(BAR_QF + s), b * 64, h, row);
      }
      issued = it + 1;
    }
    const volatile int never = 0;
    ptx::mbar_wait(bar(BAR_KV), 0, &never, p.wait_limit_ns);
    for (int it = issued > NS ? issued - NS : 0; it < issued; ++it)
      ptx::mbar_wait(bar(BAR_QF + it % NS), (it / NS) & 1, &never, p.wait_limit_ns);
  } else if (n_iter > 0 && warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop; one elected lane issues each tcgen05
    // instruction, and every wait's outcome is agreed across the warp.
    const uint32_t leader = ptx::elect_one();
    auto wait_w = [&](uint32_t b_, uint32_t parity, int where) -> bool {
      const bool w_ok = ptx::mbar_wait(b_, parity, s_abort, p.wait_limit_ns);
      if (!w_ok && leader) ptx::record_timeout(p.status, s_abort, where);
      return __all_sync(0xffffffffu, w_ok);
    };
    constexpr uint32_t idesc_s = ptx::idesc_fp16(128, 128, 0, 0);  // K-major A and B
    constexpr uint32_t idesc_kb = ptx::idesc_fp16(128, D, 0, 1);   // A K-major, B MN-major
    constexpr uint32_t idesc_q = ptx::idesc_fp16(128, D, 1, 1);    // A and B MN-major
    bool ok = wait_w(bar(BAR_KV), 0, 0x1200);
    for (int it = 0; ok && it < n_iter; ++it) {
      const int s = it % NS;
      const uint32_t q_tile = sQ + s * L::kTileBytes;
      const uint32_t do_tile = sDO + s * L::kTileBytes;
      if (!wait_w(bar(BAR_QF + s), (it / NS) & 1, 0x1300 + it)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      // S^T = K Q^T: M = keys, N = queries, K = d; both operands K-major
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
        ptx::mma_ss_w(tS, ptx::sdesc_sw128(sK + off, 16, 1024),
                         ptx::sdesc_sw128(q_tile + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u, leader);
      }
      ptx::mma_commit_w(bar(BAR_S), leader);
      if (it > 0) {
        if (!wait_w(bar(BAR_DQFREE), (it - 1) & 1, 0x1400 + it)) {
          ok = false;
          break;
        }
        ptx::tc_fence_after();
      }
      // dP^T = V dO^T
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
        ptx::mma_ss_w(tDP, ptx::sdesc_sw128(sV + off, 16, 1024),
                         ptx::sdesc_sw128(do_tile + off, 16, 1024), idesc_s, kk > 0 ? 1u : 0u, leader);
      }
      ptx::mma_commit_w(bar(BAR_DP), leader);
      if (!wait_w(bar(BAR_P), it & 1, 0x1500 + it)) {
        ok = false;
        break;
      }
      ptx::tc_fence_after();
      // dV += P^T dO and dK += dS^T Q: M = keys, N = d, K = queries.
      // A (P^T / dS^T) K-major; B (dO / Q, [queries][d]) MN-major.
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t aoff = (kk >> 2) * 16384 + (kk & 3) * 32;
        const uint32_t boff = kk * 2048;
        const uint32_t acc = (it > 0 || kk > 0) ? 1u : 0u;
        ptx::mma_ss_w(tDV, ptx::sdesc_sw128(sPt + aoff, 16, 1024),
                         ptx::sdesc_sw128(do_tile + boff, 16384, 1024), idesc_kb, acc, leader);
        ptx::mma_ss_w(tDK, ptx::sdesc_sw128(sDSt + aoff, 16, 1024),
                         ptx::sdesc_sw128(q_tile + boff, 16384, 1024), idesc_kb, acc, leader);
      }
      ptx::mma_commit_w(bar(BAR_QE + s), leader);
      // dQ = dS K: M = queries, N = d, K = keys. A = dS read from dS^T
      // ([keys][queries]) as MN-major; B = K ([keys][d]) MN-major.
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        ptx::mma_ss_w(tDP, ptx::sdesc_sw128(sDSt + kk * 2048, 16384, 1024),
                         ptx::sdesc_sw128(sK + kk * 2048, 16384, 1024), idesc_q,
                         kk > 0 ? 1u : 0u, leader);
      }
      ptx::mma_commit_w(bar(BAR_DQ), leader);
    }
    ptx::mma_commit_w(bar(BAR_DRAIN), leader);
    const volatile int never = 0;
    ptx::mbar_wait(bar(BAR_DRAIN), 0, &never, p.wait_limit_ns);
  } else if (warp < 4) {
    // ------------------------------------------------------------ compute
    const int j = threadIdx.x;  // key row (P/dS) and query row (dQ read-out)
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const int32_t kpos = kpos0 + j;
    // one past the last query that sees this key: its document end, or the
    // end of the key's sliding window when that is earlier
    const int32_t dend = p.window > 0 ? min(doc_end(p.cu, p.n_cu, kpos), kpos + p.window)
                                      : doc_end(p.cu, p.n_cu, kpos);
    bool ok = true;
    for (int it = 0; it < n_iter; ++it) {
      const int h = kh * p.G + it / n_qtiles;
      const int qt = w.lo + it % n_qtiles;
      const int64_t q_row0 = q_row_base + static_cast<int64_t>(qt) * 128;
      const int32_t qpos0 = __ldg(q_tile_pos + qt);
      float* lse2 = s_row + (it & 1) * 256;
      float* dlt = lse2 + 128;
      lse2[j] = __ldg(p.lse + static_cast<int64_t>(h) * p.T_q + q_row0 + j) * kLog2e;
      dlt[j] = __ldg(p.delta + static_cast<int64_t>(h) * p.T_q + q_row0 + j);
      // all compute threads staged their entry (bounded wait, no bar.sync,
      // so an aborting warp can never strand the others)
      ptx::mbar_arrive(bar(BAR_ROW));
      if (!ptx::mbar_wait(bar(BAR_ROW), it & 1, s_abort, p.wait_limit_ns)) {
        ptx::record_timeout(p.status, s_abort, 0x1800 + it);
        ok = false;
      }
      const bool full = (kpos0 + 127 <= qpos0) && (kpos0 >= ptx::row_lo(p.cu, p.n_cu, p.window, qpos0 + 127));
      const int lo_i = kpos - qpos0;        // first visible query column
      const int hi_i = dend - 1 - qpos0;    // last visible query column
      if (!ptx::mbar_wait(bar(BAR_S), it & 1, s_abort, p.wait_limit_ns) ||
          !ptx::mbar_wait(bar(BAR_DP), it & 1, s_abort, p.wait_limit_ns)) {
        ptx::record_timeout(p.status, s_abort, 0x1600 + it);
        ok = false;
      }
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      ptx::tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        float sv[32], dp[32];
        ptx::tmem_ld32(tS + lane_base + c * 32, sv);
        ptx::tmem_ld32(tDP + lane_base + c * 32, dp);
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          const int i = c * 32 + x;
          const bool vis = full || (i >= lo_i && i <= hi_i);
          const float pv = vis ? ptx::ex2(fmaf(sv[x], p.scale_log2, -lse2[i])) : 0.f;
          sv[x] = pv;
          dp[x] = pv * (dp[x] - dlt[i]);
        }
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const int chunk = c * 4 + ch;
          const float* a = sv + ch * 8;
          const float* b = dp + ch * 8;
          ptx::st_shared_v4(sPt + sw128_offset(j, chunk), ptx::pack_f16(a[0], a[1]),
                            ptx::pack_f16(a[2], a[3]), ptx::pack_f16(a[4], a[5]),
                            ptx::pack_f16(a[6], a[7]));
          ptx::st_shared_v4(sDSt + sw128_offset(j, chunk), ptx::pack_f16(b[0], b[1]),
                            ptx::pack_f16(b[2], b[3]), ptx::pack_f16(b[4], b[5]),
                            ptx::pack_f16(b[6], b[7]));
        }
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(BAR_P));
      if (!ptx::mbar_wait(bar(BAR_DQ), it & 1, s_abort, p.wait_limit_ns)) {
        ptx::record_timeout(p.status, s_abort, 0x1700 + it);
        ok = false;
      }
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      ptx::tc_fence_after();
      // dQ row j of this query tile: scale * (dS K)[j, :], added in fp32
      float* dq_row = p.dq + ((q_row0 + j) * p.Hq + h) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        float v[32];
        ptx::tmem_ld32(tDP + lane_base + c * 32, v);
#pragma unroll
        for (int x4 = 0; x4 < 8; ++x4) {
          float4 a = make_float4(v[x4 * 4] * p.scale, v[x4 * 4 + 1] * p.scale,
                                 v[x4 * 4 + 2] * p.scale, v[x4 * 4 + 3] * p.scale);
          atomicAdd(reinterpret_cast<float4*>(dq_row + c * 32 + x4 * 4), a);
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(BAR_DQFREE));
    }
    ok = __all_sync(0xffffffffu, ok);
    if (ok && n_iter > 0) {
      // all MMAs finished (the last BAR_DQ covers them): dK and dV rows
      float* dk_row = p.dk + ((kv_row0 + j) * p.Hkv + kh) * D;
      float* dv_row = p.dv + ((kv_row0 + j) * p.Hkv + kh) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        float a[32], b[32];
        ptx::tmem_ld32(tDK + lane_base + c * 32, a);
        ptx::tmem_ld32(tDV + lane_base + c * 32, b);
        float4* dk4 = reinterpret_cast<float4*>(dk_row + c * 32);
        float4* dv4 = reinterpret_cast<float4*>(dv_row + c * 32);
#pragma unroll
        for (int x4 = 0; x4 < 8; ++x4) {
          float4 u = dk4[x4];
          u.x += a[x4 * 4] * p.scale;
          u.y += a[x4 * 4 + 1] * p.scale;
          u.z += a[x4 * 4 + 2] * p.scale;
          u.w += a[x4 * 4 + 3] * p.scale;
          dk4[x4] = u;
          float4 t = dv4[x4];
          t.x += b[x4 * 4];
          t.y += b[x4 * 4 + 1];
          t.z += b[x4 * 4 + 2];
          t.w += b[x4 * 4 + 3];
          dv4[x4] = t;
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

// ===========================================================================
// d = 128: pipelined variant with 64-row query sub-tiles.
//
// Per iteration (one 64-row query sub-tile of one head of the group):
//   S^T  = K Q^T    (M = 128 keys, N = 64)   TMEM buffer b = it & 1
//   dP^T = V dO^T   (M = 128 keys, N = 64)   TMEM buffer b
//   P^T (fp16) -> back into buffer b's S^T columns of TMEM, dS^T (fp16) ->
//   shared-memory buffer b, by compute warpgroup b
//   dQ^T = K^T dS^T (M = 128 = d, N = 64)   TMEM, in buffer b's dP^T columns
//   dV += P^T dO (P^T read from TMEM), dK += dS^T Q   (M = 128 keys, N = 128)
// Two compute warpgroups take alternate iterations, so one warpgroup's
// exponentials and its dQ read-out overlap the other's MMAs, and both TMEM
// buffers and both shared-memory buffers alternate with them. The MMA warp
// issues S^T/dP^T of iteration it+1 before the dQ^T/dV/dK of iteration it,
// and dQ^T before dV/dK, so the read-out of dQ^T that frees a buffer runs
// while the tensor core still has dV/dK queued. dQ comes out
// transposed (TMEM lane = column of d), so each warp's fp32 reduction into
// dq covers 32 consecutive floats of one query row: one 128-byte line per
// instruction.
// Warps: 0-3 compute warpgroup 0, 4-7 compute warpgroup 1, 8 TMA producer,
// 9 TMEM owner + MMA issuer (320 threads).
// TMEM columns: buffer b: S^T (then P^T in its first 32 columns)
// [128b, 128b+64), dP^T (then dQ^T) [128b+64, 128b+128); dV [256, 384),
// dK [384, 512).
// Q/dO (and the sub-tile's LSE/delta rows) come through a 3-stage TMA ring:
// a stage is free only after that iteration's dV/dK MMAs, so two stages would
// leave the next load's latency exposed every iteration.
constexpr int kThreadsW = 320;
constexpr int kStagesW = 3;

enum : int {
  WB_KV = 0,
  WB_QF = 1,                     // [kStagesW]
  WB_QE = WB_QF + kStagesW,      // [kStagesW]
  WB_SDP = WB_QE + kStagesW,     // [2]
  WB_P = WB_SDP + 2,             // [2] 128 arrivals
  WB_DQ = WB_P + 2,              // [2]
  WB_FREE = WB_DQ + 2,           // [2] 128 arrivals
  WB_DRAIN = WB_FREE + 2,
  WB_COUNT = WB_DRAIN + 1
};

struct BwdWideSmem {
  static constexpr int kKV = 128 * 128 * 2;    // K or V tile, fp16
  static constexpr int kQT = 64 * 128 * 2;     // Q or dO sub-tile
  static constexpr int kPT = 128 * 64 * 2;     // dS^T buffer
  static constexpr int kK = 0;
  static constexpr int kV = kK + kKV;
  static constexpr int kQ = kV + kKV;                   // [kStagesW]
  static constexpr int kDO = kQ + kStagesW * kQT;       // [kStagesW]
  static constexpr int kDSt = kDO + kStagesW * kQT;     // [2]
  static constexpr int kRow = kDSt + 2 * kPT;           // [kStagesW][lse|delta][64] f32
  static constexpr int kBar = kRow + kStagesW * 2 * 64 * 4;
  static constexpr int kMisc = kBar + WB_COUNT * 8;
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kAlloc = kBytes + 1024;
};

__global__ void __launch_bounds__(kThreadsW, 1)
    step_bwd_wide_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_do, const BwdParams p) {
  using L = BwdWideSmem;
  constexpr int D = 128;
  constexpr int NS = kStagesW;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_u32 = ptx::smem_u32(smem_raw);
  const uint32_t pad = (1024u - (raw_u32 & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const uint32_t sbase = raw_u32 + pad;
  const uint32_t sK = sbase + L::kK;
  const uint32_t sV = sbase + L::kV;
  const uint32_t sQ = sbase + L::kQ;
  const uint32_t sDO = sbase + L::kDO;
  const uint32_t sDSt = sbase + L::kDSt;
  const uint32_t sRow = sbase + L::kRow;
  const float* s_row = reinterpret_cast<const float*>(smem + L::kRow);  // [stage][lse | delta][64]
  const uint32_t bar0 = sbase + L::kBar;
  auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int item = blockIdx.x / p.Hkv;
  const int kh = blockIdx.x % p.Hkv;
  const WorkItem w = p.items[item];
  const int n_sub = 2 * (w.hi - w.lo);  // 64-row query sub-tiles per head
  const int n_iter = n_sub * p.G;
  const int64_t kv_row0 = static_cast<int64_t>(w.kv_owner) * p.n_kv + static_cast<int64_t>(w.tile) * 128;
  const int32_t kpos0 = __ldg(p.kv_tile_pos + static_cast<int64_t>(w.kv_owner) * p.n_kt + w.tile);
  const int32_t* q_tile_pos = p.q_tile_pos + static_cast<int64_t>(w.q_owner) * p.n_qt;
  const int64_t q_row_base = static_cast<int64_t>(w.q_owner) * p.n_q + static_cast<int64_t>(w.lo) * 128;

  if (threadIdx.x == 0) {
    for (int i = 0; i < WB_COUNT; ++i) {
      const bool many = (i >= WB_P && i < WB_P + 2) || (i >= WB_FREE && i < WB_FREE + 2);
      ptx::mbar_init(bar(i), many ? 128u : 1u);
    }
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
  // chained after a previous step: with large GQA groups only the launch
  // overlaps its tail (see the host side)
  if (p.dep_wait_early) ptx::grid_dep_wait();
  const uint32_t tDV = tmem + 256;
  const uint32_t tDK = tmem + 384;

  if (n_iter > 0 && warp == 8 && lane == 0) {
    // ------------------------------------------------------------ producer
    ptx::prefetch_tmap(&tm_q);
    ptx::prefetch_tmap(&tm_k);
    ptx::prefetch_tmap(&tm_v);
    ptx::prefetch_tmap(&tm_do);
    ptx::mbar_arrive_expect_tx(bar(WB_KV), 2 * L::kKV);
    for (int b = 0; b < 2; ++b) {
      ptx::tma_load_3d(sK + b * 16384, &tm_k, bar(WB_KV), b * 64, kh, static_cast<int>(kv_row0));
      ptx::tma_load_3d(sV + b * 16384, &tm_v, bar(WB_KV), b * 64, kh, static_cast<int>(kv_row0));
    }
    int issued = 0;
    for (int it = 0; it < n_iter; ++it) {
      const int s = it % NS;
      if (it >= NS) {
        if (!ptx::mbar_wait(bar(WB_QE + s), ((it / NS) - 1) & 1, s_abort, p.wait_limit_ns)) {
          ptx::record_timeout(p.status, s_abort, 0x2100 + it);
          break;
        }
      }
      const int h = kh * p.G + it / n_sub;
      const int row = static_cast<int>(q_row_base + static_cast<int64_t>(it % n_sub) * 64);
      ptx::mbar_arrive_expect_tx(bar(WB_QF + s), 2 * L::kQT + 2 * 64 * 4);
      for (int b = 0; b < 2; ++b) {
        ptx::tma_load_3d(sQ + s * L::kQT + b * 8192, &tm_q, bar(WB_QF + s), b * 64, h, row);
        ptx::tma_load_3d(sDO + s * L::kQT + b * 8192, &tm_do, bar(WB_QF + s), b * 64, h, row);
      }
      // the sub-tile's 64 LSE and delta values (256 bytes each, contiguous)
      const int64_t row_off = static_cast<int64_t>(h) * p.T_q + row;
      ptx::bulk_load(sRow + s * 512, p.lse + row_off, 256, bar(WB_QF + s));
      ptx::bulk_load(sRow + s * 512 + 256, p.delta + row_off, 256, bar(WB_QF + s));
      issued = it + 1;
    }
    const volatile int never = 0;
    ptx::mbar_wait(bar(WB_KV), 0, &never, p.wait_limit_ns);
    for (int it = issued > NS ? issued - NS : 0; it < issued; ++it)
      ptx::mbar_wait(bar(WB_QF + it % NS), (it / NS) & 1, &never, p.wait_limit_ns);
  } else if (n_iter > 0 && warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop so that descriptors stay warp-uniform;
    // one elected lane issues each tcgen05 instruction.
    const uint32_t leader = ptx::elect_one();
    constexpr uint32_t idesc_sdp = ptx::idesc_fp16(128, 64, 0, 0);   // K-major A and B
    constexpr uint32_t idesc_kv = ptx::idesc_fp16(128, 128, 0, 1);   // A K-major, B MN-major
    constexpr uint32_t idesc_dq = ptx::idesc_fp16(128, 64, 1, 1);    // A and B MN-major
    // K and V as K-major A ([128][128] in two 64-column blocks of 16 KB), and
    // K as MN-major A for dQ^T (d contiguous: d 64..127 at +16 KB).
    const uint64_t dK = ptx::sdesc_sw128(sK, 16, 1024);
    const uint64_t dV = ptx::sdesc_sw128(sV, 16, 1024);
    const uint64_t dK_mn = ptx::sdesc_sw128(sK, 16384, 1024);
    auto wait_all = [&](uint32_t b_, uint32_t parity, int where) -> bool {
      const bool w_ok = ptx::mbar_wait(b_, parity, s_abort, p.wait_limit_ns);
      if (!w_ok) ptx::record_timeout(p.status, s_abort, where);
      return __all_sync(0xffffffffu, w_ok);
    };
    bool ok = wait_all(bar(WB_KV), 0, 0x2200);
    // First half of iteration it: S^T = K Q^T and dP^T = V dO^T into buffer
    // it & 1, once its Q/dO stage has landed and the buffer's previous dQ^T
    // has been read out.
    auto head = [&](int it) -> bool {
      const int b = it & 1;
      const int s = it % NS;
      {
        // the stage's Q/dO and the buffer's previous dQ^T read-out (none
        // before the third iteration: test the stage twice instead)
        const uint32_t bs[2] = {bar(WB_QF + s), it >= 2 ? bar(WB_FREE + b) : bar(WB_QF + s)};
        const uint32_t ph[2] = {static_cast<uint32_t>((it / NS) & 1),
                                it >= 2 ? static_cast<uint32_t>(((it >> 1) - 1) & 1)
                                        : static_cast<uint32_t>((it / NS) & 1)};
        if (!ptx::wait_phases(bs, ph, s_abort, p.wait_limit_ns, p.status, 0x2400 + it)) return false;
      }
      // K = d = 128; B [64][128] K-major in two blocks of 8 KB.
      const uint64_t dQk = ptx::sdesc_sw128(sQ + s * L::kQT, 16, 1024);
      const uint64_t dDOk = ptx::sdesc_sw128(sDO + s * L::kQT, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t aoff = (kk >> 2) * 16384 + (kk & 3) * 32;
        const uint32_t boff = (kk >> 2) * 8192 + (kk & 3) * 32;
        ptx::mma_ss_w(tmem + 128 * b, ptx::sdesc_add(dK, aoff), ptx::sdesc_add(dQk, boff),
                      idesc_sdp, kk > 0 ? 1u : 0u, leader);
        ptx::mma_ss_w(tmem + 128 * b + 64, ptx::sdesc_add(dV, aoff),
                      ptx::sdesc_add(dDOk, boff), idesc_sdp, kk > 0 ? 1u : 0u, leader);
      }
      ptx::mma_commit_w(bar(WB_SDP + b), leader);
      return true;
    };
    // Second half of iteration i, once its P^T and dS^T are written: dQ^T
    // first (the compute warps read it out while dV and dK run), then dV and
    // dK, after which the Q/dO stage is free.
    auto tail = [&](int i) -> bool {
      const int b = i & 1;
      const int s = i % NS;
      if (!wait_all(bar(WB_P + b), (i >> 1) & 1, 0x2300 + i)) return false;
      ptx::tc_fence_after();
      // dS^T buffer: [128 keys][64 q] fp16, one 128-byte swizzle column; read
      // K-major as A of dK and MN-major as B of dQ^T (same descriptor bits).
      const uint64_t dDS = ptx::sdesc_sw128(sDSt + b * L::kPT, 16, 1024);
      // dQ^T = K^T dS^T: M = d, N = 64 q, K = 128 keys, into the dP^T
      // columns of the buffer (already read by the compute warps).
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        ptx::mma_ss_w(tmem + 128 * b + 64, ptx::sdesc_add(dK_mn, kk * 2048),
                      ptx::sdesc_add(dDS, kk * 2048), idesc_dq, kk > 0 ? 1u : 0u, leader);
      ptx::mma_commit_w(bar(WB_DQ + b), leader);
      // Q / dO sub-tile [64 q][128 d] as MN-major B: d 64..127 at +8 KB
      const uint64_t dQm = ptx::sdesc_sw128(sQ + s * L::kQT, 8192, 1024);
      const uint64_t dDOm = ptx::sdesc_sw128(sDO + s * L::kQT, 8192, 1024);
      // dV += P^T dO (P^T read from TMEM: fp16 pairs in buffer b's first 32
      // columns, 16 queries = 8 columns) and dK += dS^T Q; K = 64 queries.
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint32_t acc = (i > 0 || kk > 0) ? 1u : 0u;
        ptx::mma_ts_w(tDV, tmem + 128 * b + kk * 8, ptx::sdesc_add(dDOm, kk * 2048), idesc_kv,
                      acc, leader);
        ptx::mma_ss_w(tDK, ptx::sdesc_add(dDS, kk * 32), ptx::sdesc_add(dQm, kk * 2048),
                      idesc_kv, acc, leader);
      }
      ptx::mma_commit_w(bar(WB_QE + s), leader);
      return true;
    };
    // S^T/dP^T of the next iteration go in before the tail of this one, so
    // that the other warpgroup computes while this tail runs.
    if (ok) ok = head(0);
    for (int it = 0; ok && it < n_iter; ++it) {
      if (it + 1 < n_iter && !head(it + 1)) { ok = false; break; }
      if (!tail(it)) { ok = false; break; }
    }
    ptx::mma_commit_w(bar(WB_DRAIN), leader);
    const volatile int never = 0;
    ptx::mbar_wait(bar(WB_DRAIN), 0, &never, p.wait_limit_ns);
    __syncwarp();
  } else if (warp < 8) {
    // ------------------------------------------------------------ compute
    const int wg = warp >> 2;                 // warpgroup = buffer parity it handles
    const int t = threadIdx.x & 127;          // key row (P/dS) and d column (dQ^T)
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int32_t kpos = kpos0 + t;
    // one past the last query that sees this key: its document end, or the
    // end of the key's sliding window when that is earlier
    const int32_t dend = p.window > 0 ? min(doc_end(p.cu, p.n_cu, kpos), kpos + p.window)
                                      : doc_end(p.cu, p.n_cu, kpos);
    const uint32_t tS = tmem + 128 * wg;
    const uint32_t tDP = tS + 64;
    const uint32_t dst = sDSt + wg * L::kPT;
    bool ok = true;
    for (int it = wg; it < n_iter; it += 2) {
      const int k = it >> 1;
      const int h = kh * p.G + it / n_sub;
      const int sub = it % n_sub;
      const int64_t q_row0 = q_row_base + static_cast<int64_t>(sub) * 64;
      const int32_t qpos0 = __ldg(q_tile_pos + w.lo + (sub >> 1)) + (sub & 1) * 64;
      // LSE and delta of the sub-tile arrive with its Q/dO stage
      const float* lse = s_row + (it % NS) * 128;
      const float* dlt = lse + 64;
      if (!ptx::mbar_wait(bar(WB_QF + it % NS), (it / NS) & 1, s_abort, p.wait_limit_ns)) {
        ptx::record_timeout(p.status, s_abort, 0x2600 + it);
        ok = false;
      }
      const bool full = (kpos0 + 127 <= qpos0) && (kpos0 >= ptx::row_lo(p.cu, p.n_cu, p.window, qpos0 + 63));
      const int lo_i = kpos - qpos0;
      const int hi_i = dend - 1 - qpos0;
      if (ok && !ptx::mbar_wait(bar(WB_SDP + wg), k & 1, s_abort, p.wait_limit_ns)) {
        ptx::record_timeout(p.status, s_abort, 0x2700 + it);
        ok = false;
      }
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      ptx::tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
        float sv[32], dp[32], l2[32], dl[32];
        ptx::tmem_ld32x2(tS + lane_base + c * 32, tDP + lane_base + c * 32, sv, dp);
        // this chunk's LSE (to base 2) and delta, 16 bytes at a time
#pragma unroll
        for (int k4 = 0; k4 < 8; ++k4) {
          const float4 a = reinterpret_cast<const float4*>(lse + c * 32)[k4];
          const float4 d4 = reinterpret_cast<const float4*>(dlt + c * 32)[k4];
          l2[4 * k4] = a.x * kLog2e;
          l2[4 * k4 + 1] = a.y * kLog2e;
          l2[4 * k4 + 2] = a.z * kLog2e;
          l2[4 * k4 + 3] = a.w * kLog2e;
          dl[4 * k4] = d4.x;
          dl[4 * k4 + 1] = d4.y;
          dl[4 * k4 + 2] = d4.z;
          dl[4 * k4 + 3] = d4.w;
        }
        if (full) {
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            const float pv = ptx::ex2(fmaf(sv[x], p.scale_log2, -l2[x]));
            sv[x] = pv;
            dp[x] = pv * (dp[x] - dl[x]);
          }
        } else {
          // branch-free mask: an invisible pair gets exponent -inf, i.e. P = 0
#pragma unroll
          for (int x = 0; x < 32; ++x) {
            const int i = c * 32 + x;
            const bool vis = i >= lo_i && i <= hi_i;
            const float arg = vis ? fmaf(sv[x], p.scale_log2, -l2[x]) : -INFINITY;
            const float pv = ptx::ex2(arg);
            sv[x] = pv;
            dp[x] = pv * (dp[x] - dl[x]);
          }
        }
        // P^T as fp16 pairs into S^T columns [16c, 16c + 16) (already read)
        uint32_t pk[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) pk[x] = ptx::pack_f16(sv[2 * x], sv[2 * x + 1]);
        ptx::tmem_st16(tS + lane_base + c * 16, pk);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          const int chunk = c * 4 + ch;  // 16-byte chunk of the 128-byte row
          const uint32_t off = static_cast<uint32_t>(t * 128 + (((chunk ^ t) & 7) << 4));
          const float* g = dp + ch * 8;
          ptx::st_shared_v4(dst + off, ptx::pack_f16(g[0], g[1]), ptx::pack_f16(g[2], g[3]),
                            ptx::pack_f16(g[4], g[5]), ptx::pack_f16(g[6], g[7]));
        }
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(WB_P + wg));
      if (!ptx::mbar_wait(bar(WB_DQ + wg), k & 1, s_abort, p.wait_limit_ns)) {
        ptx::record_timeout(p.status, s_abort, 0x2800 + it);
        ok = false;
      }
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      ptx::tc_fence_after();
      // dQ^T: lane t = column t of d; column qi = query row qi of the sub-tile.
      float* dq_col = p.dq + (q_row0 * p.Hq + h) * D + t;
      const int64_t row_stride = static_cast<int64_t>(p.Hq) * D;
      {
        float v[64];
        ptx::tmem_ld64(tDP + lane_base, v);
        // TMEM columns are free once read: let the next S^T/dP^T in
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(WB_FREE + wg));
#pragma unroll
        for (int x = 0; x < 64; ++x) atomicAdd(dq_col + x * row_stride, v[x] * p.scale);
      }
    }
    // dK (warpgroup 0) and dV (warpgroup 1) once every MMA has finished
    ok = __all_sync(0xffffffffu, ok);
    if (ok && n_iter > 0) {
      const volatile int never = 0;
      const bool done = ptx::mbar_wait(bar(WB_DRAIN), 0, &never, p.wait_limit_ns);
      if (__all_sync(0xffffffffu, done)) {
        // the previous ring step (when this grid was launched chained to it)
        // has finished its read-modify-write of the same dK / dV rows
        ptx::grid_dep_wait();
        ptx::tc_fence_after();
        // Rows leave through shared memory so that the global read-modify-
        // write is coalesced: per 32-column chunk the warp stages its 32 rows
        // (each thread its own row, 16-byte units XOR-swizzled by row), then
        // updates 4 rows per instruction, 128 contiguous bytes per row. The
        // Q/dO stages are free once every MMA has finished.
        ptx::fence_proxy_async_smem();
        float* dst = wg == 0 ? p.dk : p.dv;
        const uint32_t src = wg == 0 ? tDK : tDV;
        const float mul = wg == 0 ? p.scale : 1.f;
        uint8_t* stage = smem + L::kQ + warp * 8192;
        const int sub = lane >> 3;  // row within a group of four
        const int q4 = lane & 7;    // 16-byte unit within the chunk
        const int64_t row_stride = static_cast<int64_t>(p.Hkv) * D;
        const int64_t base_off = ((kv_row0 + (warp & 3) * 32) * p.Hkv + kh) * D + q4 * 4;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float a[32];
          ptx::tmem_ld32(src + lane_base + c * 32, a);
          uint8_t* buf = stage + (c & 1) * 4096;
#pragma unroll
          for (int x4 = 0; x4 < 8; ++x4)
            *reinterpret_cast<float4*>(buf + lane * 128 + ((x4 ^ (lane & 7)) << 4)) =
                make_float4(a[4 * x4] * mul, a[4 * x4 + 1] * mul, a[4 * x4 + 2] * mul,
                            a[4 * x4 + 3] * mul);
          __syncwarp();
          float4 old[8];
#pragma unroll
          for (int it = 0; it < 8; ++it)
            old[it] = *reinterpret_cast<const float4*>(dst + base_off + (it * 4 + sub) * row_stride + c * 32);
#pragma unroll
          for (int it = 0; it < 8; ++it) {
            const int row = it * 4 + sub;
            const float4 t4 = *reinterpret_cast<const float4*>(buf + row * 128 + ((q4 ^ (row & 7)) << 4));
            const float4 v = make_float4(old[it].x + t4.x, old[it].y + t4.y, old[it].z + t4.z,
                                         old[it].w + t4.w);
            *reinterpret_cast<float4*>(dst + base_off + row * row_stride + c * 32) = v;
          }
        }
      } else {
        ptx::record_timeout(p.status, s_abort, 0x2900);
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

size_t step_bwd_smem_bytes(int d) {
  return d == 128 ? BwdWideSmem::kAlloc : BwdSmem<64>::kAlloc;
}

int step_bwd_q_box_rows(int d) { return d == 128 ? 64 : 128; }

cp_attn_status launch_step_bwd(int d, dim3 grid, size_t smem, cudaStream_t s,
                               const CUtensorMap& tq, const CUtensorMap& tk,
                               const CUtensorMap& tv, const CUtensorMap& tdo,
                               const BwdParams& p, bool chained) {
  static bool attr_done[2] = {false, false};
  cudaError_t err;
  if (d == 128) {
    if (!attr_done[1]) {
      err = cudaFuncSetAttribute(step_bwd_wide_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
      if (err != cudaSuccess) return fail(CP_ATTN_ERR_CUDA, std::string("step_bwd attr: ") + cudaGetErrorString(err));
      attr_done[1] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreadsW);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = chained ? 1 : 0;
    err = cudaLaunchKernelEx(&cfg, step_bwd_wide_kernel, tq, tk, tv, tdo, p);
    if (err != cudaSuccess) return fail(CP_ATTN_ERR_CUDA, std::string("step_bwd launch: ") + cudaGetErrorString(err));
  } else {
    if (!attr_done[0]) {
      err = cudaFuncSetAttribute(step_bwd_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(smem));
      if (err != cudaSuccess) return fail(CP_ATTN_ERR_CUDA, std::string("step_bwd attr: ") + cudaGetErrorString(err));
      attr_done[0] = true;
    }
    step_bwd_kernel<64><<<grid, kThreads, smem, s>>>(tq, tk, tv, tdo, p);
  }
  err = cudaGetLastError();
  if (err != cudaSuccess) return fail(CP_ATTN_ERR_CUDA, std::string("step_bwd launch: ") + cudaGetErrorString(err));
  count_launch();
  return CP_ATTN_OK;
}

}  // namespace cpa
