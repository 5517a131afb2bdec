// Kernel parameter blocks and host-side launchers of the ring-attention step.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace cpa {

// Default limit of every pipeline wait inside a kernel (nanoseconds).
constexpr uint64_t kWaitLimitNs = 1000000000ull;

struct FwdParams {
  const WorkItem* items;
  const int32_t* q_tile_pos;  // [R][n_qt] first global position of each q tile
  const int32_t* kv_tile_pos; // [R][n_kt]
  const int32_t* cu;          // document offsets
  int n_cu;                   // n_docs + 1
  int32_t window;             // sliding window in tokens, 0 = none
  int n_qt, n_kt;
  int64_t n_q, n_kv, T_q;
  int Hq, G;
  float scale_log2;           // softmax scale * log2(e)
  int mode;                   // cp_attn_merge_mode
  int first;                  // ACCUMULATE: initialise the accumulators
  int part_bf16;              // WRITE_PARTIAL: o_part holds bf16 partials
  float* o_part;
  float* lse_part;
  __nv_bfloat16* o_final;     // optional
  const float* scales;        // E4M3 kernel: device [3] descale factors of q, k, v
  int32_t* status;
  uint64_t wait_limit_ns;
};

struct BwdParams {
  const WorkItem* items;
  const int32_t* q_tile_pos;
  const int32_t* kv_tile_pos;
  const int32_t* cu;
  int n_cu;
  int32_t window;             // sliding window in tokens, 0 = none
  int n_qt, n_kt;
  int64_t n_q, n_kv, T_q, T_kv;
  int Hq, Hkv, G;
  float scale;                // softmax scale
  float scale_log2;
  const float* lse;           // [Hq, T_q] natural log
  const float* delta;         // [Hq, T_q]
  float* dq;                  // [T_q, Hq, d]
  float* dk;                  // [T_kv, Hkv, d]
  float* dv;
  int32_t* status;
  uint64_t wait_limit_ns;
  // chained launch: wait for the previous step before the main loop instead
  // of before the dK / dV read-modify-write
  int dep_wait_early;
};

// chained: launch with programmatic stream serialization, so that the grid
// may start while the kernel before it (the previous ring step) drains; the
// d = 128 kernels wait for it before their accumulator read-modify-write.
cp_attn_status launch_step_fwd(int d, dim3 grid, size_t smem, cudaStream_t s,
                               const CUtensorMap& tq, const CUtensorMap& tk,
                               const CUtensorMap& tv, const FwdParams& p, bool chained);
size_t step_fwd_smem_bytes(int d);

// E4M3 forward step (head_dim 128): q, k E4M3 [tokens][heads][128] maps
// (128-byte boxes), tvt the V^T map E4M3 [heads][128][tokens]; p.scales set.
cp_attn_status launch_step_fwd_fp8(dim3 grid, size_t smem, cudaStream_t s,
                                   const CUtensorMap& tq, const CUtensorMap& tk,
                                   const CUtensorMap& tvt, const FwdParams& p, bool chained);
size_t step_fwd_fp8_smem_bytes();

// Per-tensor E4M3 quantization (fp8.cu). absmax: *amax_bits = bits of
// max |x| over n bf16 values (n a multiple of 8; zeroed first on the stream).
cp_attn_status launch_fp8_absmax(const void* x, int64_t n, unsigned int* amax_bits,
                                 cudaStream_t s);
// quantize: x bf16 [rows][heads][d] -> E4M3 in the same layout, or (transpose)
// [heads][d][rows] with rows a multiple of 64; *scale (if not NULL) gets the
// descale factor amax / 448.
cp_attn_status launch_fp8_quantize(const void* x, int64_t rows, int heads, int d,
                                   const unsigned int* amax_bits, int transpose, void* out,
                                   float* scale, cudaStream_t s);
// Query heads one forward CTA handles (d = 128 pairs the heads of a group).
int step_fwd_heads_per_cta(int d);

cp_attn_status launch_step_bwd(int d, dim3 grid, size_t smem, cudaStream_t s,
                               const CUtensorMap& tq, const CUtensorMap& tk,
                               const CUtensorMap& tv, const CUtensorMap& tdo,
                               const BwdParams& p, bool chained);
size_t step_bwd_smem_bytes(int d);
// Rows of the Q / dO tensor-map box the backward kernel for head_dim d uses.
int step_bwd_q_box_rows(int d);

// o_parts: fp32, or bf16 when parts_bf16 (part_stride in elements). pdl:
// the merge of few (row, head) pairs over many parts is launched as a
// programmatic dependent of the previous kernel on s, and waits for it before
// it reads anything.
cp_attn_status launch_merge_lse(int n_parts, int64_t rows, int heads, int d,
                                const void* o_parts, int64_t part_stride,
                                const float* lse_parts, int64_t lse_part_stride,
                                __nv_bfloat16* o_out, float* o_out_f32, float* lse_out,
                                cudaStream_t s, bool parts_bf16 = false, bool pdl = false);

// K6: n fp32 values -> bf16 (round to nearest even); n a multiple of 8,
// both pointers 16-byte aligned.
cp_attn_status launch_f32_to_bf16(const float* in, void* out, int64_t n, cudaStream_t s);

// Sequence <-> head all-to-all (gather = 0: split heads, 1: gather them).
cp_attn_status launch_head_a2a(int64_t rows, int heads, int64_t head_bytes, int a2a, int gather,
                               const void* in, void* out, cudaStream_t s);

cp_attn_status launch_permute_rows(const int32_t* row_map, int64_t rows, int64_t row_bytes,
                                   int to_natural, const void* in, void* out, cudaStream_t s);

// O from o_f32 when it is not null, else from the bf16 o.
cp_attn_status launch_bwd_preprocess(int64_t rows, int heads, int d, const __nv_bfloat16* o,
                                     const float* o_f32, const __nv_bfloat16* dout,
                                     float* delta, cudaStream_t s);

cp_attn_status launch_zero_f32(float* p, int64_t n, cudaStream_t s);

// [rows, heads, d] bf16 tensor map, 64 x 1 x 128 boxes, 128-byte swizzle (api.cu).
cp_attn_status encode_bf16_rows_map(CUtensorMap* m, const void* base, int64_t rows, int heads,
                                    int d);
// One-byte tensor map: [rows, heads, d] with d x 1 x 128 boxes, or transposed
// [heads, d, rows] with 128 x d x 1 boxes; 128-byte swizzle (api.cu).
cp_attn_status encode_u8_map(CUtensorMap* m, const void* base, int64_t rows, int heads, int d,
                             bool transposed);

cp_attn_status launch_selftest_wait(int32_t* status, uint64_t limit_ns, cudaStream_t s);

// n = element count, a multiple of 8
cp_attn_status launch_bf16_to_f16(const void* in, void* out, int64_t n, int32_t* status,
                                  cudaStream_t s);

}  // namespace cpa
