// C ABI of the ring-attention step library: argument checks, plan upload,
// tensor-map encoding and the emulated ring driver (an ordered loop of step
// launches on the caller's stream).
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <string>

#include "kernels.h"

namespace cpa {

namespace {
thread_local std::string g_err;
std::atomic<int64_t> g_launches{0};

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
    cudaGetLastError();
  });
  return fn;
}

// [rows, heads, d] bf16 viewed as a 3-D tensor (d, heads, rows); boxes of
// 64 x 1 x 128 elements land in shared memory as 128 rows of 128 bytes with
// the 128-byte swizzle.
cp_attn_status tmap_3d(CUtensorMap* m, const void* base, int64_t rows, int heads, int d,
                       CUtensorMapDataType dtype, int box_rows = 128) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(CP_ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(heads),
                              static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2,
                                 static_cast<cuuint64_t>(heads) * d * 2};
  const cuuint32_t box[3] = {64, 1, static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, dtype, 3, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(CP_ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed with code " + std::to_string(r));
  return CP_ATTN_OK;
}

cp_attn_status tmap_bf16(CUtensorMap* m, const void* base, int64_t rows, int heads, int d) {
  return tmap_3d(m, base, rows, heads, d, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
}

// One-byte elements. rows layout: [rows][heads][d] viewed as (d, heads, rows)
// with a box of d x 1 x 128; transposed layout: [heads][d][rows] viewed as
// (rows, d, heads) with a box of 128 x d x 1. Either box lands in shared
// memory as 128-byte rows with the 128-byte swizzle (d = 128).
cp_attn_status tmap_u8(CUtensorMap* m, const void* base, int64_t rows, int heads, int d,
                       bool transposed) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(CP_ATTN_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  cuuint64_t dims[3];
  cuuint64_t strides[2];
  cuuint32_t box[3];
  if (!transposed) {
    dims[0] = static_cast<cuuint64_t>(d);
    dims[1] = static_cast<cuuint64_t>(heads);
    dims[2] = static_cast<cuuint64_t>(rows);
    strides[0] = static_cast<cuuint64_t>(d);
    strides[1] = static_cast<cuuint64_t>(heads) * d;
    box[0] = static_cast<cuuint32_t>(d);
    box[1] = 1;
    box[2] = 128;
  } else {
    dims[0] = static_cast<cuuint64_t>(rows);
    dims[1] = static_cast<cuuint64_t>(d);
    dims[2] = static_cast<cuuint64_t>(heads);
    strides[0] = static_cast<cuuint64_t>(rows);
    strides[1] = static_cast<cuuint64_t>(rows) * d;
    box[0] = 128;
    box[1] = static_cast<cuuint32_t>(d);
    box[2] = 1;
  }
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(CP_ATTN_ERR_CUDA, "cuTensorMapEncodeTiled failed with code " + std::to_string(r));
  return CP_ATTN_OK;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Offsets of the fp16 copies of q, k, v, dout inside the half-operand buffer.
struct HalfOps {
  size_t q, k, v, dout, total;
};
HalfOps half_ops_layout(const cp_attn_plan_s* p) {
  HalfOps h;
  const size_t qb = round256(static_cast<size_t>(p->T_q) * p->Hq * p->d * 2);
  const size_t kb = round256(static_cast<size_t>(p->T_kv) * p->Hkv * p->d * 2);
  h.q = 0;
  h.k = qb;
  h.v = qb + kb;
  h.dout = qb + 2 * kb;
  h.total = 2 * qb + 2 * kb;
  return h;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

cp_attn_status check_device_plan(const cp_attn_plan_s* p) {
  if (!p) return fail(CP_ATTN_ERR_INVALID_ARG, "null plan");
  if (!p->on_device)
    return fail(CP_ATTN_ERR_CUDA, "plan has no device tables (no CUDA device when it was built)");
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != p->device)
    return fail(CP_ATTN_ERR_INVALID_ARG, "plan was built on CUDA device " +
                                             std::to_string(p->device) +
                                             " but another device is current");
  return CP_ATTN_OK;
}

template <typename T>
cp_attn_status upload(T** dst, const T* src, size_t n) {
  if (n == 0) n = 1;
  if (cudaMalloc(reinterpret_cast<void**>(dst), n * sizeof(T)) != cudaSuccess) {
    cudaGetLastError();
    *dst = nullptr;
    return fail(CP_ATTN_ERR_OOM, "plan: cudaMalloc of device tables failed");
  }
  if (src && cudaMemcpy(*dst, src, n * sizeof(T), cudaMemcpyHostToDevice) != cudaSuccess)
    return fail(CP_ATTN_ERR_CUDA, "plan: copy of device tables failed");
  return CP_ATTN_OK;
}

}  // namespace

cp_attn_status fail(cp_attn_status s, const std::string& msg) {
  g_err = msg;
  return s;
}
void clear_error() { g_err.clear(); }
void count_launch(int n) { g_launches += n; }

cp_attn_status upload_plan(cp_attn_plan_s* p) {
  int count = 0;
  if (cudaGetDeviceCount(&count) != cudaSuccess || count == 0) {
    cudaGetLastError();
    p->on_device = false;
    return CP_ATTN_OK;
  }
  if (cudaGetDevice(&p->device) != cudaSuccess) {
    cudaGetLastError();
    p->on_device = false;
    return CP_ATTN_OK;
  }
  std::vector<int32_t> row_q(p->q_pos.size()), row_kv(p->kv_pos.size());
  // natural query row of position x: sequence b = x / (P + N), then its new
  // token x - b (P + N) - P
  const int64_t seq = p->P + p->N;
  for (size_t i = 0; i < row_q.size(); ++i) {
    const int64_t b = p->q_pos[i] / seq;
    row_q[i] = static_cast<int32_t>(b * p->N + (p->q_pos[i] - b * seq - p->P));
  }
  for (size_t i = 0; i < row_kv.size(); ++i) row_kv[i] = static_cast<int32_t>(p->kv_pos[i]);
  const int32_t zeros[kStatusWords] = {0, 0, 0, 0};
  cp_attn_status st;
  if ((st = upload(&p->d_q_tile_pos, p->q_tile_pos.data(), p->q_tile_pos.size())) != CP_ATTN_OK ||
      (st = upload(&p->d_kv_tile_pos, p->kv_tile_pos.data(), p->kv_tile_pos.size())) != CP_ATTN_OK ||
      (st = upload(&p->d_cu, p->cu.data(), p->cu.size())) != CP_ATTN_OK ||
      (st = upload(&p->d_fwd, p->fwd_items.data(), p->fwd_items.size())) != CP_ATTN_OK ||
      (st = upload(&p->d_bwd, p->bwd_items.data(), p->bwd_items.size())) != CP_ATTN_OK ||
      (st = upload(&p->d_status, zeros, kStatusWords)) != CP_ATTN_OK ||
      (st = upload(&p->d_row_q, row_q.data(), row_q.size())) != CP_ATTN_OK ||
      (st = upload(&p->d_row_kv, row_kv.data(), row_kv.size())) != CP_ATTN_OK) {
    free_plan_device(p);
    return st;
  }
  const size_t v16_bytes = static_cast<size_t>(p->T_kv) * p->Hkv * p->d * 2;
  if (cudaMalloc(&p->d_v16, v16_bytes > 0 ? v16_bytes : 16) != cudaSuccess) {
    cudaGetLastError();
    p->d_v16 = nullptr;
    free_plan_device(p);
    return fail(CP_ATTN_ERR_OOM, "plan: cannot allocate the fp16 copy of V (" +
                                     std::to_string(v16_bytes) + " bytes)");
  }
  p->on_device = true;
  return CP_ATTN_OK;
}

void free_plan_device(cp_attn_plan_s* p) {
  void* ptrs[] = {p->d_q_tile_pos, p->d_kv_tile_pos, p->d_cu,    p->d_fwd,  p->d_bwd,
                  p->d_status,      p->d_row_q,       p->d_row_kv, p->d_v16};
  for (void* q : ptrs)
    if (q) cudaFree(q);
  p->d_q_tile_pos = p->d_kv_tile_pos = p->d_cu = p->d_status = p->d_row_q = p->d_row_kv = nullptr;
  p->d_v16 = nullptr;
  p->d_fwd = p->d_bwd = nullptr;
  p->on_device = false;
}

// [rows, heads, d] bf16 tensor map with 64 x 1 x 128 boxes (the step kernels'
// view), for kernels outside this file.
cp_attn_status encode_bf16_rows_map(CUtensorMap* m, const void* base, int64_t rows, int heads,
                                    int d) {
  return tmap_bf16(m, base, rows, heads, d);
}

// One-byte [rows, heads, d] map (128-byte boxes), or the transposed
// [heads, d, rows] one (128 x d boxes), for kernels outside this file.
cp_attn_status encode_u8_map(CUtensorMap* m, const void* base, int64_t rows, int heads, int d,
                             bool transposed) {
  return tmap_u8(m, base, rows, heads, d, transposed);
}

}  // namespace cpa

using namespace cpa;

extern "C" {

const char* cp_attn_last_error(void) { return g_err.c_str(); }

const char* cp_attn_status_string(cp_attn_status s) {
  switch (s) {
    case CP_ATTN_OK: return "ok";
    case CP_ATTN_ERR_INVALID_ARG: return "invalid argument";
    case CP_ATTN_ERR_SHAPE: return "bad shape";
    case CP_ATTN_ERR_UNSUPPORTED: return "unsupported";
    case CP_ATTN_ERR_CUDA: return "CUDA error";
    case CP_ATTN_ERR_OOM: return "out of device memory";
    case CP_ATTN_ERR_TIMEOUT: return "kernel wait timed out";
    case CP_ATTN_ERR_RANGE: return "input value out of the supported range";
  }
  return "unknown status";
}

int64_t cp_attn_launch_count(void) { return g_launches.load(); }

cp_attn_status cp_attn_plan_ex(cp_attn_plan_t* out, const cp_attn_plan_desc* desc) {
  clear_error();
  if (!out) return fail(CP_ATTN_ERR_INVALID_ARG, "plan: null output handle");
  *out = nullptr;
  auto* p = new (std::nothrow) cp_attn_plan_s();
  if (!p) return fail(CP_ATTN_ERR_OOM, "plan: host allocation failed");
  cp_attn_status st = build_plan(p, desc);
  if (st == CP_ATTN_OK) st = upload_plan(p);
  if (st != CP_ATTN_OK) {
    delete p;
    return st;
  }
  *out = p;
  return CP_ATTN_OK;
}

cp_attn_status cp_attn_plan(cp_attn_plan_t* out, int64_t seq_len, int cp, int n_q_heads,
                            int n_kv_heads, int head_dim, cp_attn_layout layout,
                            cp_attn_variant variant, const int32_t* cu_seqlens, int n_docs) {
  cp_attn_plan_desc d;
  std::memset(&d, 0, sizeof(d));
  d.seq_len = seq_len;
  d.kv_prefix_len = 0;
  d.cp = cp;
  d.n_q_heads = n_q_heads;
  d.n_kv_heads = n_kv_heads;
  d.head_dim = head_dim;
  d.layout = layout;
  d.variant = variant;
  d.cu_seqlens = cu_seqlens;
  d.n_docs = n_docs;
  d.softmax_scale = 0.f;
  return cp_attn_plan_ex(out, &d);
}

void cp_attn_plan_destroy(cp_attn_plan_t plan) {
  if (!plan) return;
  free_plan_device(plan);
  delete plan;
}

cp_attn_status cp_attn_select_variant(int64_t n_new, int64_t n_cached, int n_q_heads,
                                      int n_kv_heads, cp_attn_variant* out) {
  clear_error();
  if (!out || n_new <= 0 || n_cached < 0 || n_q_heads <= 0 || n_kv_heads <= 0)
    return fail(CP_ATTN_ERR_INVALID_ARG, "select_variant: bad arguments");
  *out = select_variant_rule(n_new, n_cached, n_q_heads, n_kv_heads);
  return CP_ATTN_OK;
}

cp_attn_status cp_attn_plan_info(cp_attn_plan_t p, int64_t* info, int n) {
  clear_error();
  if (!p || !info || n < 0 || n > 16) return fail(CP_ATTN_ERR_INVALID_ARG, "plan_info: bad arguments");
  const int64_t v[16] = {p->T_q, p->T_kv, p->n_q, p->n_kv, p->R, p->Hq, p->Hkv, p->d,
                         p->n_qt, p->n_kt, static_cast<int64_t>(p->cu.size()) - 1,
                         p->on_device ? 1 : 0, static_cast<int64_t>(p->variant), p->window,
                         p->a2a, p->B};
  for (int i = 0; i < n; ++i) info[i] = v[i];
  return CP_ATTN_OK;
}

cp_attn_status cp_attn_plan_work_list(cp_attn_plan_t p, int step, int backward, int32_t* out,
                                      int64_t* n_items) {
  clear_error();
  if (!p || !n_items || step < 0 || step >= p->R || (backward != 0 && backward != 1))
    return fail(CP_ATTN_ERR_INVALID_ARG, "plan_work_list: bad arguments");
  const std::vector<cpa::WorkItem>& items = backward ? p->bwd_items : p->fwd_items;
  const std::vector<int>& off = backward ? p->bwd_off : p->fwd_off;
  const int a = off[step], b = off[step + 1];
  *n_items = b - a;
  if (out) {
    for (int i = a; i < b; ++i) {
      const cpa::WorkItem& w = items[i];
      int32_t* o = out + static_cast<int64_t>(i - a) * 6;
      o[0] = w.q_owner;
      o[1] = w.kv_owner;
      o[2] = w.tile;
      o[3] = w.lo;
      o[4] = w.hi;
      o[5] = w.n_full;
    }
  }
  return CP_ATTN_OK;
}

cp_attn_status cp_attn_plan_positions(cp_attn_plan_t p, cp_attn_tensor_kind kind, int rank,
                                      int32_t* out) {
  clear_error();
  if (!p || !out || rank < 0 || rank >= p->R)
    return fail(CP_ATTN_ERR_INVALID_ARG, "plan_positions: bad arguments");
  if (kind == CP_ATTN_TENSOR_Q) {
    for (int64_t i = 0; i < p->n_q; ++i) out[i] = static_cast<int32_t>(p->q_pos[rank * p->n_q + i]);
  } else if (kind == CP_ATTN_TENSOR_KV) {
    for (int64_t i = 0; i < p->n_kv; ++i) out[i] = static_cast<int32_t>(p->kv_pos[rank * p->n_kv + i]);
  } else {
    return fail(CP_ATTN_ERR_INVALID_ARG, "plan_positions: bad tensor kind");
  }
  return CP_ATTN_OK;
}

cp_attn_status cp_attn_plan_schedule(cp_attn_plan_t p, int32_t* out) {
  clear_error();
  if (!p || !out) return fail(CP_ATTN_ERR_INVALID_ARG, "plan_schedule: bad arguments");
  std::memcpy(out, p->sched.data(), p->sched.size() * sizeof(int32_t));
  return CP_ATTN_OK;
}

cp_attn_status cp_attn_plan_block_mask(cp_attn_plan_t p, uint8_t* out) {
  clear_error();
  if (!p || !out) return fail(CP_ATTN_ERR_INVALID_ARG, "plan_block_mask: bad arguments");
  size_t idx = 0;
  for (int a = 0; a < p->R; ++a)
    for (int b = 0; b < p->R; ++b)
      for (int i = 0; i < p->n_qt; ++i)
        for (int j = 0; j < p->n_kt; ++j) out[idx++] = static_cast<uint8_t>(tile_class(p, a, i, b, j));
  return CP_ATTN_OK;
}

cp_attn_status cp_attn_plan_visible_pairs(cp_attn_plan_t p, int step, int64_t* out) {
  clear_error();
  if (!p || !out || step < -1 || step >= p->R)
    return fail(CP_ATTN_ERR_INVALID_ARG, "plan_visible_pairs: bad arguments");
  if (step >= 0) {
    *out = p->step_pairs[step];
  } else {
    int64_t s = 0;
    for (int64_t v : p->step_pairs) s += v;
    *out = s;
  }
  return CP_ATTN_OK;
}

namespace {

// Pass-Q forward workspace: R O partial slots (fp32 or bf16), then R fp32
// LSE slots.
struct PassQLayout {
  int64_t o_slot, l_slot;  // elements per slot
  size_t lse_off, total;   // bytes
};
PassQLayout pass_q_layout(cp_attn_plan_t p) {
  PassQLayout L;
  L.o_slot = p->T_q * p->Hq * p->d;
  L.l_slot = p->T_q * p->Hq;
  const size_t elt = p->part_bf16 ? 2 : 4;
  L.lse_off = round256(static_cast<size_t>(L.o_slot) * p->R * elt);
  L.total = L.lse_off + round256(static_cast<size_t>(L.l_slot) * p->R * sizeof(float));
  return L;
}

// Backward workspace: delta, the fp16 operand copies, then (bf16 gradients)
// the fp32 accumulators of dq, dk, dv.
struct BwdLayout {
  size_t half_ops, dq, dk, dv, total;  // byte offsets, size
};
BwdLayout bwd_layout(cp_attn_plan_t p) {
  BwdLayout L;
  L.half_ops = round256(static_cast<size_t>(p->T_q) * p->Hq * sizeof(float));
  L.dq = L.half_ops + half_ops_layout(p).total;
  const size_t nq = static_cast<size_t>(p->T_q) * p->Hq * p->d * sizeof(float);
  const size_t nk = static_cast<size_t>(p->T_kv) * p->Hkv * p->d * sizeof(float);
  L.dk = L.dq + (p->grad_bf16 ? round256(nq) : 0);
  L.dv = L.dk + (p->grad_bf16 ? round256(nk) : 0);
  L.total = L.dv + (p->grad_bf16 ? round256(nk) : 0);
  return L;
}

}  // namespace

cp_attn_status cp_attn_workspace_size(cp_attn_plan_t p, cp_attn_op op, size_t* bytes) {
  clear_error();
  if (!p || !bytes) return fail(CP_ATTN_ERR_INVALID_ARG, "workspace_size: bad arguments");
  const size_t o = static_cast<size_t>(p->T_q) * p->Hq * p->d * sizeof(float);
  if (op == CP_ATTN_OP_FORWARD) {
    *bytes = p->variant == CP_ATTN_PASS_KV ? round256(o) : pass_q_layout(p).total;
  } else if (op == CP_ATTN_OP_BACKWARD) {
    *bytes = bwd_layout(p).total;
  } else {
    return fail(CP_ATTN_ERR_INVALID_ARG, "workspace_size: bad op");
  }
  return CP_ATTN_OK;
}

cp_attn_status cp_attn_half_ops_size(cp_attn_plan_t p, size_t* bytes) {
  clear_error();
  if (!p || !bytes) return fail(CP_ATTN_ERR_INVALID_ARG, "half_ops_size: bad arguments");
  *bytes = half_ops_layout(p).total;
  return CP_ATTN_OK;
}

namespace {

// One forward ring step. chained: launch it so that it may overlap the tail of
// the kernel before it, which must be an earlier step of the same ring.
// *launched tells whether a kernel went out (a step without work launches none).
// scales != NULL selects the E4M3 kernel: q, k E4M3 [T][H][128], v then
// holds V^T E4M3 [Hkv][128][T_kv], scales the device descale factors.
cp_attn_status step_fwd_impl(cp_attn_plan_t p, int step, const void* q, const void* k,
                             const void* v, void* o_part, float* lse_part,
                             cp_attn_merge_mode mode, void* o_final, void* stream, bool chained,
                             bool* launched, const float* scales = nullptr) {
  *launched = false;
  cp_attn_status st = check_device_plan(p);
  if (st != CP_ATTN_OK) return st;
  if (step < 0 || step >= p->R) return fail(CP_ATTN_ERR_INVALID_ARG, "step_fwd: step out of range");
  if (mode != CP_ATTN_WRITE_PARTIAL && mode != CP_ATTN_ACCUMULATE)
    return fail(CP_ATTN_ERR_INVALID_ARG, "step_fwd: bad merge mode");
  if (!q || !k || !v || !o_part || !lse_part)
    return fail(CP_ATTN_ERR_INVALID_ARG, "step_fwd: null tensor pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o_part) ||
      (o_final && !aligned16(o_final)))
    return fail(CP_ATTN_ERR_INVALID_ARG, "step_fwd: tensors must be 16-byte aligned");
  const bool fp8 = scales != nullptr;
  if (fp8 && p->d != 128)
    return fail(CP_ATTN_ERR_UNSUPPORTED, "step_fwd_fp8: head_dim must be 128");
  if (fp8 && !aligned16(scales))
    return fail(CP_ATTN_ERR_INVALID_ARG, "step_fwd_fp8: scales must be 16-byte aligned");
  CUtensorMap tq, tk, tv;
  if (fp8) {
    if ((st = tmap_u8(&tq, q, p->T_q, p->Hq, p->d, false)) != CP_ATTN_OK) return st;
    if ((st = tmap_u8(&tk, k, p->T_kv, p->Hkv, p->d, false)) != CP_ATTN_OK) return st;
    if ((st = tmap_u8(&tv, v, p->T_kv, p->Hkv, p->d, true)) != CP_ATTN_OK) return st;
  } else {
    // the ring's first step copies V to fp16 for the P V products of every
    // step (P then keeps 11 significant bits)
    if (step == 0 &&
        (st = launch_bf16_to_f16(v, p->d_v16, p->T_kv * p->Hkv * p->d, p->d_status,
                                 static_cast<cudaStream_t>(stream))) != CP_ATTN_OK)
      return st;
    if ((st = tmap_bf16(&tq, q, p->T_q, p->Hq, p->d)) != CP_ATTN_OK) return st;
    if ((st = tmap_bf16(&tk, k, p->T_kv, p->Hkv, p->d)) != CP_ATTN_OK) return st;
    if ((st = tmap_3d(&tv, p->d_v16, p->T_kv, p->Hkv, p->d, CU_TENSOR_MAP_DATA_TYPE_FLOAT16)) !=
        CP_ATTN_OK)
      return st;
  }
  FwdParams fp;
  std::memset(&fp, 0, sizeof(fp));
  fp.items = p->d_fwd + p->fwd_off[step];
  fp.q_tile_pos = p->d_q_tile_pos;
  fp.kv_tile_pos = p->d_kv_tile_pos;
  fp.cu = p->d_cu;
  fp.n_cu = static_cast<int>(p->cu.size());
  fp.window = static_cast<int32_t>(p->window);
  fp.n_qt = p->n_qt;
  fp.n_kt = p->n_kt;
  fp.n_q = p->n_q;
  fp.n_kv = p->n_kv;
  fp.T_q = p->T_q;
  fp.Hq = p->Hq;
  fp.G = p->Hq / p->Hkv;
  fp.scale_log2 = p->scale * 1.44269504088896340736f;
  fp.mode = mode;
  fp.first = (mode == CP_ATTN_ACCUMULATE && step == 0) ? 1 : 0;
  fp.part_bf16 = (mode == CP_ATTN_WRITE_PARTIAL && p->part_bf16) ? 1 : 0;
  fp.o_part = static_cast<float*>(o_part);
  fp.lse_part = lse_part;
  fp.o_final = mode == CP_ATTN_ACCUMULATE ? static_cast<__nv_bfloat16*>(o_final) : nullptr;
  fp.scales = scales;
  fp.status = p->d_status;
  fp.wait_limit_ns = kWaitLimitNs;
  // Items without visible tiles still run when every row must be written:
  // partial outputs, accumulator initialisation, or the final bf16 output.
  const bool all_items = (mode == CP_ATTN_WRITE_PARTIAL) || fp.first || fp.o_final != nullptr;
  const int n_items = all_items ? (p->fwd_off[step + 1] - p->fwd_off[step]) : p->fwd_nonempty[step];
  if (n_items == 0) return CP_ATTN_OK;
  *launched = true;
  // one CTA per (item, query head), or per (item, pair of heads of a group)
  const int hpc = step_fwd_heads_per_cta(p->d);
  const int G = p->Hq / p->Hkv;
  const int64_t units = hpc == 1 ? p->Hq : static_cast<int64_t>(p->Hkv) * ((G + 1) / 2);
  const dim3 grid(static_cast<unsigned>(static_cast<int64_t>(n_items) * units));
  if (fp8)
    return launch_step_fwd_fp8(grid, step_fwd_fp8_smem_bytes(), static_cast<cudaStream_t>(stream),
                               tq, tk, tv, fp, chained);
  return launch_step_fwd(p->d, grid, step_fwd_smem_bytes(p->d), static_cast<cudaStream_t>(stream),
                         tq, tk, tv, fp, chained);
}

// One backward ring step; chained and *launched as for step_fwd_impl.
cp_attn_status step_bwd_impl(cp_attn_plan_t p, int step, const void* half_ops, const float* lse,
                             const float* delta, float* dq_acc, float* dk_acc, float* dv_acc,
                             void* stream, bool chained, bool* launched) {
  *launched = false;
  cp_attn_status st = check_device_plan(p);
  if (st != CP_ATTN_OK) return st;
  if (step < 0 || step >= p->R) return fail(CP_ATTN_ERR_INVALID_ARG, "step_bwd: step out of range");
  if (!half_ops || !lse || !delta || !dq_acc || !dk_acc || !dv_acc)
    return fail(CP_ATTN_ERR_INVALID_ARG, "step_bwd: null tensor pointer");
  if ((reinterpret_cast<uintptr_t>(half_ops) & 255u) || !aligned16(dq_acc) ||
      !aligned16(dk_acc) || !aligned16(dv_acc) || !aligned16(lse) || !aligned16(delta))
    return fail(CP_ATTN_ERR_INVALID_ARG,
                "step_bwd: half_ops must be 256-byte aligned; accumulators, lse and delta "
                "16-byte aligned");
  const HalfOps ho = half_ops_layout(p);
  const char* hb = static_cast<const char*>(half_ops);
  CUtensorMap tq, tk, tv, tdo;
  const CUtensorMapDataType f16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const int qbox = step_bwd_q_box_rows(p->d);
  if ((st = tmap_3d(&tq, hb + ho.q, p->T_q, p->Hq, p->d, f16, qbox)) != CP_ATTN_OK) return st;
  if ((st = tmap_3d(&tk, hb + ho.k, p->T_kv, p->Hkv, p->d, f16)) != CP_ATTN_OK) return st;
  if ((st = tmap_3d(&tv, hb + ho.v, p->T_kv, p->Hkv, p->d, f16)) != CP_ATTN_OK) return st;
  if ((st = tmap_3d(&tdo, hb + ho.dout, p->T_q, p->Hq, p->d, f16, qbox)) != CP_ATTN_OK) return st;
  BwdParams bp;
  std::memset(&bp, 0, sizeof(bp));
  bp.items = p->d_bwd + p->bwd_off[step];
  bp.q_tile_pos = p->d_q_tile_pos;
  bp.kv_tile_pos = p->d_kv_tile_pos;
  bp.cu = p->d_cu;
  bp.n_cu = static_cast<int>(p->cu.size());
  bp.window = static_cast<int32_t>(p->window);
  bp.n_qt = p->n_qt;
  bp.n_kt = p->n_kt;
  bp.n_q = p->n_q;
  bp.n_kv = p->n_kv;
  bp.T_q = p->T_q;
  bp.T_kv = p->T_kv;
  bp.Hq = p->Hq;
  bp.Hkv = p->Hkv;
  bp.G = p->Hq / p->Hkv;
  bp.scale = p->scale;
  bp.scale_log2 = p->scale * 1.44269504088896340736f;
  bp.lse = lse;
  bp.delta = delta;
  bp.dq = dq_acc;
  bp.dk = dk_acc;
  bp.dv = dv_acc;
  bp.status = p->d_status;
  bp.wait_limit_ns = kWaitLimitNs;
  // Measured on GB300: letting a chained step's main loop run beside the
  // previous step's tail gains ~2 % with up to 8 query heads per KV head and
  // loses up to 17 % with 16 (the 405B-shaped and packed 128/8-head layers),
  // so larger groups wait before the loop and only the launch overlaps.
  bp.dep_wait_early = (p->Hq / p->Hkv > 8) ? 1 : 0;
  const int n_items = p->bwd_off[step + 1] - p->bwd_off[step];
  if (n_items == 0) return CP_ATTN_OK;
  *launched = true;
  const dim3 grid(static_cast<unsigned>(static_cast<int64_t>(n_items) * p->Hkv));
  return launch_step_bwd(p->d, grid, step_bwd_smem_bytes(p->d), static_cast<cudaStream_t>(stream),
                         tq, tk, tv, tdo, bp, chained);
}

}  // namespace

cp_attn_status cp_attn_step_fwd(cp_attn_plan_t p, int step, const void* q, const void* k,
                                const void* v, void* o_part, float* lse_part,
                                cp_attn_merge_mode mode, void* o_final, void* stream) {
  clear_error();
  bool launched = false;
  return step_fwd_impl(p, step, q, k, v, o_part, lse_part, mode, o_final, stream,
                       p && p->chain_steps && step > 0, &launched);
}

cp_attn_status cp_attn_step_bwd_half(cp_attn_plan_t p, int step, const void* half_ops,
                                     const float* lse, const float* delta, float* dq_acc,
                                     float* dk_acc, float* dv_acc, void* stream) {
  clear_error();
  bool launched = false;
  return step_bwd_impl(p, step, half_ops, lse, delta, dq_acc, dk_acc, dv_acc, stream,
                       p && p->chain_steps && step > 0, &launched);
}

cp_attn_status cp_attn_step_bwd(cp_attn_plan_t p, int step, const void* q, const void* k,
                                const void* v, const void* dout, const float* lse,
                                const float* delta, float* dq_acc, float* dk_acc,
                                float* dv_acc, void* workspace, size_t workspace_bytes,
                                void* stream) {
  clear_error();
  cp_attn_status st = check_device_plan(p);
  if (st != CP_ATTN_OK) return st;
  if (step < 0 || step >= p->R) return fail(CP_ATTN_ERR_INVALID_ARG, "step_bwd: step out of range");
  if (!q || !k || !v || !dout || !workspace)
    return fail(CP_ATTN_ERR_INVALID_ARG, "step_bwd: null pointer");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dout))
    return fail(CP_ATTN_ERR_INVALID_ARG, "step_bwd: q, k, v, dout must be 16-byte aligned");
  const HalfOps ho = half_ops_layout(p);
  if (workspace_bytes < ho.total)
    return fail(CP_ATTN_ERR_INVALID_ARG, "step_bwd: workspace smaller than cp_attn_half_ops_size");
  if (reinterpret_cast<uintptr_t>(workspace) & 255u)
    return fail(CP_ATTN_ERR_INVALID_ARG, "step_bwd: workspace must be 256-byte aligned");
  if (step == 0) {
    // the ring's first step makes the fp16 operand copies every step reads
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* hb = static_cast<char*>(workspace);
    const int64_t nq = p->T_q * p->Hq * p->d, nk = p->T_kv * p->Hkv * p->d;
    if ((st = launch_bf16_to_f16(q, hb + ho.q, nq, p->d_status, s)) != CP_ATTN_OK) return st;
    if ((st = launch_bf16_to_f16(k, hb + ho.k, nk, p->d_status, s)) != CP_ATTN_OK) return st;
    if ((st = launch_bf16_to_f16(v, hb + ho.v, nk, p->d_status, s)) != CP_ATTN_OK) return st;
    if ((st = launch_bf16_to_f16(dout, hb + ho.dout, nq, p->d_status, s)) != CP_ATTN_OK)
      return st;
  }
  bool launched = false;
  return step_bwd_impl(p, step, workspace, lse, delta, dq_acc, dk_acc, dv_acc, stream,
                       p->chain_steps && step > 0, &launched);
}

cp_attn_status cp_attn_plan_set_chaining(cp_attn_plan_t p, int enable) {
  clear_error();
  if (!p) return fail(CP_ATTN_ERR_INVALID_ARG, "plan_set_chaining: null plan");
  if (enable != 0 && enable != 1) return fail(CP_ATTN_ERR_INVALID_ARG, "plan_set_chaining: enable must be 0 or 1");
  p->chain_steps = enable;
  return CP_ATTN_OK;
}

cp_attn_status cp_attn_step_fwd_fp8(cp_attn_plan_t p, int step, const void* q8, const void* k8,
                                    const void* vt8, const float* scales, void* o_part,
                                    float* lse_part, cp_attn_merge_mode mode, void* o_final,
                                    void* stream) {
  clear_error();
  if (!scales) return fail(CP_ATTN_ERR_INVALID_ARG, "step_fwd_fp8: null scales");
  bool launched = false;
  return step_fwd_impl(p, step, q8, k8, vt8, o_part, lse_part, mode, o_final, stream,
                       p && p->chain_steps && step > 0, &launched, scales);
}

cp_attn_status cp_attn_fp8_absmax(const void* x, int64_t n, float* amax, void* stream) {
  clear_error();
  if (!x || !amax) return fail(CP_ATTN_ERR_INVALID_ARG, "fp8_absmax: null pointer");
  if (n < 0 || n % 8) return fail(CP_ATTN_ERR_SHAPE, "fp8_absmax: n must be a non-negative multiple of 8");
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(amax) & 3u))
    return fail(CP_ATTN_ERR_INVALID_ARG, "fp8_absmax: x must be 16-byte and amax 4-byte aligned");
  return launch_fp8_absmax(x, n, reinterpret_cast<unsigned int*>(amax),
                           static_cast<cudaStream_t>(stream));
}

cp_attn_status cp_attn_fp8_quantize(const void* x, int64_t rows, int heads, int head_dim,
                                    const float* amax, int transpose, void* out, float* scale,
                                    void* stream) {
  clear_error();
  if (!x || !amax || !out) return fail(CP_ATTN_ERR_INVALID_ARG, "fp8_quantize: null pointer");
  if (rows < 0 || heads <= 0 || (head_dim != 64 && head_dim != 128))
    return fail(CP_ATTN_ERR_SHAPE, "fp8_quantize: head_dim must be 64 or 128, heads positive");
  if (transpose != 0 && transpose != 1)
    return fail(CP_ATTN_ERR_INVALID_ARG, "fp8_quantize: transpose must be 0 or 1");
  if (transpose && rows % 64)
    return fail(CP_ATTN_ERR_SHAPE, "fp8_quantize: transposed output needs rows % 64 == 0");
  if (!aligned16(x) || !aligned16(out) || (reinterpret_cast<uintptr_t>(amax) & 3u) ||
      (reinterpret_cast<uintptr_t>(scale) & 3u))
    return fail(CP_ATTN_ERR_INVALID_ARG, "fp8_quantize: misaligned pointer");
  return launch_fp8_quantize(x, rows, heads, head_dim,
                             reinterpret_cast<const unsigned int*>(amax), transpose, out, scale,
                             static_cast<cudaStream_t>(stream));
}

cp_attn_status cp_attn_bwd_preprocess(cp_attn_plan_t p, const void* q, const void* k,
                                      const void* v, const void* o, const float* o_f32,
                                      const void* dout, float* delta, void* half_ops,
                                      float* dq_acc, float* dk_acc, float* dv_acc,
                                      void* stream) {
  clear_error();
  cp_attn_status st = check_device_plan(p);
  if (st != CP_ATTN_OK) return st;
  if ((half_ops && (!q || !k || !v)) || (!o && !o_f32) || !dout || !delta)
    return fail(CP_ATTN_ERR_INVALID_ARG, "bwd_preprocess: null pointer");
  if ((q && !aligned16(q)) || (k && !aligned16(k)) || (v && !aligned16(v)) ||
      (o && !aligned16(o)) ||
      (o_f32 && !aligned16(o_f32)) || !aligned16(dout) ||
      (reinterpret_cast<uintptr_t>(half_ops) & 255u) || (dq_acc && !aligned16(dq_acc)) ||
      (dk_acc && !aligned16(dk_acc)) || (dv_acc && !aligned16(dv_acc)))
    return fail(CP_ATTN_ERR_INVALID_ARG, "bwd_preprocess: misaligned pointer");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = launch_bwd_preprocess(p->T_q, p->Hq, p->d, static_cast<const __nv_bfloat16*>(o),
                                  o_f32, static_cast<const __nv_bfloat16*>(dout), delta, s)) !=
      CP_ATTN_OK)
    return st;
  const HalfOps ho = half_ops_layout(p);
  char* hb = static_cast<char*>(half_ops);
  const int64_t nq = p->T_q * p->Hq * p->d, nk = p->T_kv * p->Hkv * p->d;
  if (half_ops) {
    if ((st = launch_bf16_to_f16(q, hb + ho.q, nq, p->d_status, s)) != CP_ATTN_OK) return st;
    if ((st = launch_bf16_to_f16(k, hb + ho.k, nk, p->d_status, s)) != CP_ATTN_OK) return st;
    if ((st = launch_bf16_to_f16(v, hb + ho.v, nk, p->d_status, s)) != CP_ATTN_OK) return st;
    if ((st = launch_bf16_to_f16(dout, hb + ho.dout, nq, p->d_status, s)) != CP_ATTN_OK)
      return st;
  }
  if (dq_acc && (st = launch_zero_f32(dq_acc, nq, s)) != CP_ATTN_OK) return st;
  if (dk_acc && (st = launch_zero_f32(dk_acc, nk, s)) != CP_ATTN_OK) return st;
  if (dv_acc && (st = launch_zero_f32(dv_acc, nk, s)) != CP_ATTN_OK) return st;
  return CP_ATTN_OK;
}

cp_attn_status cp_attn_merge_lse_ex(int n_parts, int64_t rows, int heads, int head_dim,
                                    cp_attn_dtype parts_dtype, const void* o_parts,
                                    int64_t part_stride, const float* lse_parts,
                                    int64_t lse_part_stride, void* o_out, float* o_out_f32,
                                    float* lse_out, void* stream) {
  clear_error();
  if (n_parts < 1 || rows < 0 || heads < 1 || head_dim < 4 || head_dim % 4 || head_dim > 256)
    return fail(CP_ATTN_ERR_SHAPE, "merge_lse: bad sizes");
  if (parts_dtype != CP_ATTN_F32 && parts_dtype != CP_ATTN_BF16)
    return fail(CP_ATTN_ERR_INVALID_ARG, "merge_lse: parts_dtype must be F32 or BF16");
  if (!o_parts || !lse_parts || !lse_out)
    return fail(CP_ATTN_ERR_INVALID_ARG, "merge_lse: null pointer");
  if (!aligned16(o_parts) || (part_stride % 4) || (o_out && (reinterpret_cast<uintptr_t>(o_out) & 7)) ||
      (o_out_f32 && !aligned16(o_out_f32)))
    return fail(CP_ATTN_ERR_INVALID_ARG, "merge_lse: misaligned pointer or stride");
  const bool bf16 = parts_dtype == CP_ATTN_BF16;
  if (bf16 && o_out_f32) {
    // the fp32 output may not overlap the bf16 parts (they are read by other blocks)
    const char* a = static_cast<const char*>(o_parts);
    const char* b = reinterpret_cast<const char*>(o_out_f32);
    const int64_t span = ((n_parts - 1) * part_stride + rows * heads * head_dim) * 2;
    if (b < a + span && a < b + rows * heads * head_dim * 4)
      return fail(CP_ATTN_ERR_INVALID_ARG, "merge_lse: o_out_f32 overlaps bf16 parts");
  }
  return launch_merge_lse(n_parts, rows, heads, head_dim, o_parts, part_stride, lse_parts,
                          lse_part_stride, static_cast<__nv_bfloat16*>(o_out), o_out_f32, lse_out,
                          static_cast<cudaStream_t>(stream), bf16);
}

cp_attn_status cp_attn_merge_lse(int n_parts, int64_t rows, int heads, int head_dim,
                                 const float* o_parts, int64_t part_stride,
                                 const float* lse_parts, int64_t lse_part_stride, void* o_out,
                                 float* o_out_f32, float* lse_out, void* stream) {
  return cp_attn_merge_lse_ex(n_parts, rows, heads, head_dim, CP_ATTN_F32, o_parts, part_stride,
                              lse_parts, lse_part_stride, o_out, o_out_f32, lse_out, stream);
}

cp_attn_status cp_attn_forward(cp_attn_plan_t p, const void* q, const void* k, const void* v,
                               void* o, float* lse, void* workspace, size_t workspace_bytes,
                               void* stream) {
  clear_error();
  cp_attn_status st = check_device_plan(p);
  if (st != CP_ATTN_OK) return st;
  size_t need = 0;
  cp_attn_workspace_size(p, CP_ATTN_OP_FORWARD, &need);
  if (!workspace || workspace_bytes < need)
    return fail(CP_ATTN_ERR_INVALID_ARG, "forward: workspace smaller than cp_attn_workspace_size");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(CP_ATTN_ERR_INVALID_ARG, "forward: workspace must be 256-byte aligned");
  if (!o || !lse) return fail(CP_ATTN_ERR_INVALID_ARG, "forward: null output");
  float* ws = static_cast<float*>(workspace);
  if (p->variant == CP_ATTN_PASS_KV) {
    // Q stays, KV moves; merge "as it goes" into the fp32 accumulator
    // each step after the first that launches overlaps the tail of the one before
    bool prev = false;
    for (int t = 0; t < p->R; ++t) {
      bool launched = false;
      st = step_fwd_impl(p, t, q, k, v, ws, lse, CP_ATTN_ACCUMULATE, t == p->R - 1 ? o : nullptr,
                         stream, prev, &launched);
      if (st != CP_ATTN_OK) return st;
      prev = prev || launched;
    }
    return CP_ATTN_OK;
  }
  // Pass Q: KV stays, Q moves. Each step writes its partials to the slot of
  // the kv owner (the permutation back to order); the n-way merge per q owner
  // stands for the all-to-all plus merge.
  const PassQLayout L = pass_q_layout(p);
  float* ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + L.lse_off);
  bool prev = false;
  for (int t = 0; t < p->R; ++t) {
    bool launched = false;
    st = step_fwd_impl(p, t, q, k, v, ws, ws_lse, CP_ATTN_WRITE_PARTIAL, nullptr, stream, prev,
                       &launched);
    if (st != CP_ATTN_OK) return st;
    prev = prev || launched;
  }
  // The merge also leaves the fp32 result in slot 0 (each (row, head) is read
  // completely by one warp before that warp writes it); bf16 slots are too
  // small for it.
  return cp_attn_merge_lse_ex(p->R, p->T_q, p->Hq, p->d, p->part_bf16 ? CP_ATTN_BF16 : CP_ATTN_F32,
                              ws, L.o_slot, ws_lse, L.l_slot, o, p->part_bf16 ? nullptr : ws, lse,
                              stream);
}

cp_attn_status cp_attn_forward_fp8(cp_attn_plan_t p, const void* q8, const void* k8,
                                   const void* vt8, const float* scales, void* o, float* lse,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  cp_attn_status st = check_device_plan(p);
  if (st != CP_ATTN_OK) return st;
  if (!scales) return fail(CP_ATTN_ERR_INVALID_ARG, "forward_fp8: null scales");
  size_t need = 0;
  cp_attn_workspace_size(p, CP_ATTN_OP_FORWARD, &need);
  if (!workspace || workspace_bytes < need)
    return fail(CP_ATTN_ERR_INVALID_ARG, "forward_fp8: workspace smaller than cp_attn_workspace_size");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(CP_ATTN_ERR_INVALID_ARG, "forward_fp8: workspace must be 256-byte aligned");
  if (!o || !lse) return fail(CP_ATTN_ERR_INVALID_ARG, "forward_fp8: null output");
  float* ws = static_cast<float*>(workspace);
  bool prev = false;
  if (p->variant == CP_ATTN_PASS_KV) {
    for (int t = 0; t < p->R; ++t) {
      bool launched = false;
      st = step_fwd_impl(p, t, q8, k8, vt8, ws, lse, CP_ATTN_ACCUMULATE,
                         t == p->R - 1 ? o : nullptr, stream, prev, &launched, scales);
      if (st != CP_ATTN_OK) return st;
      prev = prev || launched;
    }
    return CP_ATTN_OK;
  }
  const PassQLayout L = pass_q_layout(p);
  float* ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + L.lse_off);
  for (int t = 0; t < p->R; ++t) {
    bool launched = false;
    st = step_fwd_impl(p, t, q8, k8, vt8, ws, ws_lse, CP_ATTN_WRITE_PARTIAL, nullptr, stream,
                       prev, &launched, scales);
    if (st != CP_ATTN_OK) return st;
    prev = prev || launched;
  }
  return cp_attn_merge_lse_ex(p->R, p->T_q, p->Hq, p->d, p->part_bf16 ? CP_ATTN_BF16 : CP_ATTN_F32,
                              ws, L.o_slot, ws_lse, L.l_slot, o, p->part_bf16 ? nullptr : ws, lse,
                              stream);
}

cp_attn_status cp_attn_backward(cp_attn_plan_t p, const void* q, const void* k, const void* v,
                                const void* o, const float* o_f32, const float* lse,
                                const void* dout, void* dq, void* dk, void* dv,
                                void* workspace, size_t workspace_bytes, void* stream) {
  clear_error();
  cp_attn_status st = check_device_plan(p);
  if (st != CP_ATTN_OK) return st;
  size_t need = 0;
  cp_attn_workspace_size(p, CP_ATTN_OP_BACKWARD, &need);
  if (!workspace || workspace_bytes < need)
    return fail(CP_ATTN_ERR_INVALID_ARG, "backward: workspace smaller than cp_attn_workspace_size");
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return fail(CP_ATTN_ERR_INVALID_ARG, "backward: workspace must be 256-byte aligned");
  if (!dq || !dk || !dv) return fail(CP_ATTN_ERR_INVALID_ARG, "backward: null gradient");
  if (!aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(CP_ATTN_ERR_INVALID_ARG, "backward: gradients must be 16-byte aligned");
  const BwdLayout L = bwd_layout(p);
  char* wb = static_cast<char*>(workspace);
  float* delta = reinterpret_cast<float*>(wb);
  void* half_ops = wb + L.half_ops;
  // bf16 gradients: the fp32 sums live in the workspace until the finalize
  float* dq_acc = p->grad_bf16 ? reinterpret_cast<float*>(wb + L.dq) : static_cast<float*>(dq);
  float* dk_acc = p->grad_bf16 ? reinterpret_cast<float*>(wb + L.dk) : static_cast<float*>(dk);
  float* dv_acc = p->grad_bf16 ? reinterpret_cast<float*>(wb + L.dv) : static_cast<float*>(dv);
  if ((st = cp_attn_bwd_preprocess(p, q, k, v, o, o_f32, dout, delta, half_ops, dq_acc, dk_acc,
                                   dv_acc, stream)) != CP_ATTN_OK)
    return st;
  bool prev = false;
  for (int t = 0; t < p->R; ++t) {
    bool launched = false;
    st = step_bwd_impl(p, t, half_ops, lse, delta, dq_acc, dk_acc, dv_acc, stream, prev,
                       &launched);
    if (st != CP_ATTN_OK) return st;
    prev = prev || launched;
  }
  if (!p->grad_bf16) return CP_ATTN_OK;
  // K6: the summed gradients rounded to bf16
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t nq = p->T_q * p->Hq * p->d, nk = p->T_kv * p->Hkv * p->d;
  if ((st = launch_f32_to_bf16(dq_acc, dq, nq, s)) != CP_ATTN_OK) return st;
  if ((st = launch_f32_to_bf16(dk_acc, dk, nk, s)) != CP_ATTN_OK) return st;
  return launch_f32_to_bf16(dv_acc, dv, nk, s);
}

cp_attn_status cp_attn_layout_apply(cp_attn_plan_t p, cp_attn_tensor_kind kind,
                                    cp_attn_direction direction, const void* in, void* out,
                                    int64_t row_bytes, void* stream) {
  clear_error();
  cp_attn_status st = check_device_plan(p);
  if (st != CP_ATTN_OK) return st;
  if (!in || !out || in == out) return fail(CP_ATTN_ERR_INVALID_ARG, "layout_apply: bad pointers");
  if (row_bytes <= 0 || row_bytes % 16) return fail(CP_ATTN_ERR_SHAPE, "layout_apply: row_bytes must be a positive multiple of 16");
  if (!aligned16(in) || !aligned16(out)) return fail(CP_ATTN_ERR_INVALID_ARG, "layout_apply: pointers must be 16-byte aligned");
  if (direction != CP_ATTN_TO_RANK_MAJOR && direction != CP_ATTN_TO_NATURAL)
    return fail(CP_ATTN_ERR_INVALID_ARG, "layout_apply: bad direction");
  const int32_t* map;
  int64_t rows;
  if (kind == CP_ATTN_TENSOR_Q) {
    map = p->d_row_q;
    rows = p->T_q;
  } else if (kind == CP_ATTN_TENSOR_KV) {
    map = p->d_row_kv;
    rows = p->T_kv;
  } else {
    return fail(CP_ATTN_ERR_INVALID_ARG, "layout_apply: bad tensor kind");
  }
  return launch_permute_rows(map, rows, row_bytes, direction == CP_ATTN_TO_NATURAL ? 1 : 0, in, out,
                             static_cast<cudaStream_t>(stream));
}

cp_attn_status cp_attn_head_a2a(int64_t rows, int heads, int64_t head_bytes, int a2a,
                                cp_attn_a2a_direction direction, const void* in, void* out,
                                void* stream) {
  clear_error();
  if (!in || !out) return fail(CP_ATTN_ERR_INVALID_ARG, "head_a2a: null pointer");
  if (rows < 0 || heads <= 0 || a2a <= 0 || heads % a2a != 0)
    return fail(CP_ATTN_ERR_SHAPE, "head_a2a: heads must be a positive multiple of a2a");
  if (head_bytes <= 0 || head_bytes % 16)
    return fail(CP_ATTN_ERR_SHAPE, "head_a2a: head_bytes must be a positive multiple of 16");
  if (!aligned16(in) || !aligned16(out))
    return fail(CP_ATTN_ERR_INVALID_ARG, "head_a2a: pointers must be 16-byte aligned");
  if (direction != CP_ATTN_SPLIT_HEADS && direction != CP_ATTN_GATHER_HEADS)
    return fail(CP_ATTN_ERR_INVALID_ARG, "head_a2a: bad direction");
  const int64_t bytes = rows * heads * head_bytes;
  const char* ci = static_cast<const char*>(in);
  const char* co = static_cast<const char*>(out);
  if (ci < co + bytes && co < ci + bytes)
    return fail(CP_ATTN_ERR_INVALID_ARG, "head_a2a: in and out overlap");
  return launch_head_a2a(rows, heads, head_bytes, a2a, direction == CP_ATTN_GATHER_HEADS ? 1 : 0,
                         in, out, static_cast<cudaStream_t>(stream));
}

cp_attn_status cp_attn_selftest_wait_timeout(cp_attn_plan_t p, uint64_t limit_ns, void* stream) {
  clear_error();
  cp_attn_status st = check_device_plan(p);
  if (st != CP_ATTN_OK) return st;
  if (limit_ns == 0 || limit_ns > 2000000000ull)
    return fail(CP_ATTN_ERR_INVALID_ARG, "selftest_wait_timeout: limit must be in (0, 2 s]");
  return launch_selftest_wait(p->d_status, limit_ns, static_cast<cudaStream_t>(stream));
}

cp_attn_status cp_attn_sync_status(cp_attn_plan_t p, void* stream) {
  clear_error();
  cp_attn_status st = check_device_plan(p);
  if (st != CP_ATTN_OK) return st;
  cudaError_t err = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (err != cudaSuccess) return fail(CP_ATTN_ERR_CUDA, std::string("sync: ") + cudaGetErrorString(err));
  int32_t host[kStatusWords] = {0, 0, 0, 0};
  err = cudaMemcpy(host, p->d_status, sizeof(host), cudaMemcpyDeviceToHost);
  if (err != cudaSuccess) return fail(CP_ATTN_ERR_CUDA, std::string("status read: ") + cudaGetErrorString(err));
  if (host[0] != 0) {
    const int32_t zeros[kStatusWords] = {0, 0, 0, 0};
    cudaMemcpy(p->d_status, zeros, sizeof(zeros), cudaMemcpyHostToDevice);
    return fail(static_cast<cp_attn_status>(host[0]),
                "device status " + std::to_string(host[0]) + " in block " + std::to_string(host[1]) +
                    " at 0x" + [&] { char b[16]; std::snprintf(b, sizeof(b), "%x", host[2]); return std::string(b); }());
  }
  return CP_ATTN_OK;
}

}  // extern "C"
