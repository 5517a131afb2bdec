// Internal declarations shared by the host planner, the C-ABI layer and the
// kernels of the ring-attention step library.
#pragma once

#include <cstddef>
#include <cstdint>
#include <string>
#include <vector>

#include "cp_attn.h"

namespace cpa {

constexpr int kTile = 128;  // query rows and keys per tile

// One unit of kernel work. Forward: q tile `tile` of rank q_owner against the
// kv tiles [lo, hi) of rank kv_owner. Backward: kv tile `tile` of rank
// kv_owner against the q tiles [lo, hi) of rank q_owner. Every tile in
// [lo, hi) is non-empty (positions are increasing in local order, so the
// visible tiles of a tile form one run).
struct WorkItem {
  int32_t q_owner;
  int32_t kv_owner;
  int32_t tile;
  int32_t lo;
  int32_t hi;
  int32_t n_full;  // tiles of [lo, hi) that are FULL (no element mask)
  int32_t pad0;
  int32_t pad1;
};
static_assert(sizeof(WorkItem) == 32, "WorkItem layout");

// Device status word layout: [0] error code, [1] block, [2] role/where.
constexpr int kStatusWords = 4;

}  // namespace cpa

struct cp_attn_plan_s {
  // description
  int64_t N = 0;   // new tokens
  int64_t P = 0;   // cached prefix
  int64_t B = 1;   // independent sequences (each P + N tokens)
  int R = 0, Hq = 0, Hkv = 0, d = 0;
  cp_attn_layout layout = CP_ATTN_LAYOUT_ZIGZAG;
  int a2a = 1;              // USP all-to-all group size
  cp_attn_variant variant = CP_ATTN_PASS_KV;
  float scale = 0.f;
  int64_t window = 0;       // sliding window in tokens, 0 = none
  std::vector<int32_t> cu;  // document offsets (at least {0, P+N})
  // sizes
  int64_t n_q = 0, n_kv = 0, T_q = 0, T_kv = 0;
  int n_qt = 0, n_kt = 0;
  // positions (rank-major)
  std::vector<int64_t> q_pos, kv_pos;            // [R*n_q], [R*n_kv]
  std::vector<int32_t> q_tile_pos, kv_tile_pos;  // [R*n_qt], [R*n_kt]
  std::vector<int32_t> sched;                    // [R][R][2]
  // work lists, concatenated over steps
  std::vector<cpa::WorkItem> fwd_items, bwd_items;
  std::vector<int> fwd_off, fwd_nonempty;  // per step: offset, non-empty count
  std::vector<int> bwd_off;                // per step offset (all non-empty)
  std::vector<int64_t> step_pairs;         // visible pairs per step per q head
  // device copies
  bool on_device = false;
  int device = -1;
  int32_t* d_q_tile_pos = nullptr;
  int32_t* d_kv_tile_pos = nullptr;
  int32_t* d_cu = nullptr;
  cpa::WorkItem* d_fwd = nullptr;
  cpa::WorkItem* d_bwd = nullptr;
  int32_t* d_status = nullptr;
  int32_t* d_row_q = nullptr;   // rank-major row -> natural row (queries)
  int32_t* d_row_kv = nullptr;  // rank-major row -> natural row (keys)
  // fp16 copy of V [T_kv][Hkv][d], made by step 0 of every bf16 forward ring:
  // the P V products of the step kernels run on fp16 operands
  void* d_v16 = nullptr;
  // per-step calls of steps >= 1 launch chained to the kernel before them
  int chain_steps = 0;
  int part_bf16 = 0;        // WRITE_PARTIAL O partials (and Pass-Q slots) in bf16
  int grad_bf16 = 0;        // cp_attn_backward hands out bf16 gradients
};

namespace cpa {

// error reporting (thread-local message)
cp_attn_status fail(cp_attn_status s, const std::string& msg);
void clear_error();

// planner (plan.cpp)
cp_attn_status build_plan(cp_attn_plan_s* p, const cp_attn_plan_desc* desc);
int64_t doc_start_host(const std::vector<int32_t>& cu, int64_t pos);
// First key visible to the query at `pos` (document start or window start).
int64_t row_lo_host(const cp_attn_plan_s* p, int64_t pos);
// Pass Q iff its ring message (the new tokens' Q) is smaller than Pass KV's
// (K and V of all tokens).
cp_attn_variant select_variant_rule(int64_t n_new, int64_t n_cached, int hq, int hkv);
int tile_class(const cp_attn_plan_s* p, int qa_rank, int qt, int kb_rank, int kt);
int64_t tile_visible_pairs(const cp_attn_plan_s* p, int qa_rank, int qt, int kb_rank,
                           int kt);

// device upload / free (api.cu)
cp_attn_status upload_plan(cp_attn_plan_s* p);
void free_plan_device(cp_attn_plan_s* p);

// launch counter
void count_launch(int n = 1);

}  // namespace cpa
