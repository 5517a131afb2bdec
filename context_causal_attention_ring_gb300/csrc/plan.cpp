// Host planner: chunk plan, ring schedule, 128x128 block classes and the
// per-step work lists of the ring-attention step.
//
// Chunk plan: "Context Parallelism for Scalable Million-Token Inference",
// section "Load Balancing in CP" (2R chunks, rank r takes chunks r and
// 2R-1-r; the same sharding for partial prefill). Ring schedule: section
// "Ring Attention Algorithms" (Pass KV moves KV, Pass Q moves Q; at step t
// rank r holds the moving tensor of rank (r - t) mod R). Block skipping and
// packed sequences: "Announcing Long-Context Training on TPUs with MaxText
// Context Parallelism", section "Built on a fast attention kernel".
//
// Block classes use a closed form on the contiguous position ranges of a
// tile (every tile lies inside one chunk because chunks are multiples of 128
// tokens). A query q sees the keys in [lo(q), q], where lo(q) is the start of
// q's document, or q - W + 1 with a sliding window of W tokens when that is
// later (the window masks of the models that "mix sliding-window and global
// layers", section "What's next" of the MaxText post). lo is nondecreasing in
// q, so for queries [qa, qb] and keys [ka, kb], with q* = max(qa, ka):
//   non-empty  <=>  q* <= qb  and  lo(q*) <= kb
//   full       <=>  kb <= qa  and  ka >= lo(qb)
// (without a window, lo(q*) <= kb reduces to ds(qa) <= kb.)
#include <algorithm>
#include <cmath>
#include <cstring>
#include <numeric>

#include "internal.h"

namespace cpa {

int64_t doc_start_host(const std::vector<int32_t>& cu, int64_t pos) {
  // largest cu[i] <= pos
  auto it = std::upper_bound(cu.begin(), cu.end(), static_cast<int32_t>(pos));
  return static_cast<int64_t>(*(it - 1));
}

static void shard(int64_t n_tokens, int R, cp_attn_layout layout, int a2a, int64_t offset,
                  int r, std::vector<int64_t>& out) {
  if (layout == CP_ATTN_LAYOUT_ZIGZAG || layout == CP_ATTN_LAYOUT_USP) {
    // USP: ring rank r pools the zigzag pairs of devices r*a2a .. r*a2a+a2a-1
    // of D = a2a*R devices, in ascending position order: chunks
    // r*a2a .. r*a2a+a2a-1, then 2D-r*a2a-a2a .. 2D-1-r*a2a (zigzag is the
    // case a2a = 1)
    const int64_t U = layout == CP_ATTN_LAYOUT_USP ? a2a : 1;
    const int64_t D = U * R;
    const int64_t c = n_tokens / (2 * D);
    for (int half = 0; half < 2; ++half)
      for (int64_t u = 0; u < U; ++u) {
        const int64_t ch = half == 0 ? r * U + u : 2 * D - r * U - U + u;
        for (int64_t i = 0; i < c; ++i) out.push_back(offset + ch * c + i);
      }
  } else {
    const int64_t c = n_tokens / R;
    for (int64_t i = 0; i < c; ++i) out.push_back(offset + r * c + i);
  }
}

int64_t row_lo_host(const cp_attn_plan_s* p, int64_t pos) {
  const int64_t ds = doc_start_host(p->cu, pos);
  return p->window > 0 ? std::max(ds, pos - p->window + 1) : ds;
}

cp_attn_variant select_variant_rule(int64_t n_new, int64_t n_cached, int hq, int hkv) {
  // Pass Q sends T_new*Hq*d elements per hop, Pass KV 2*T_total*Hkv*d.
  const double q_msg = static_cast<double>(n_new) * hq;
  const double kv_msg = 2.0 * static_cast<double>(n_new + n_cached) * hkv;
  return q_msg < kv_msg ? CP_ATTN_PASS_Q : CP_ATTN_PASS_KV;
}

int tile_class(const cp_attn_plan_s* p, int qr, int qt, int kr, int kt) {
  const int64_t qa = p->q_tile_pos[static_cast<size_t>(qr) * p->n_qt + qt];
  const int64_t qb = qa + kTile - 1;
  const int64_t ka = p->kv_tile_pos[static_cast<size_t>(kr) * p->n_kt + kt];
  const int64_t kb = ka + kTile - 1;
  const int64_t qs = std::max(qa, ka);
  if (!(qs <= qb && row_lo_host(p, qs) <= kb)) return 0;
  if (kb <= qa && ka >= row_lo_host(p, qb)) return 2;
  return 1;
}

int64_t tile_visible_pairs(const cp_attn_plan_s* p, int qr, int qt, int kr, int kt) {
  const int cls = tile_class(p, qr, qt, kr, kt);
  if (cls == 0) return 0;
  if (cls == 2) return static_cast<int64_t>(kTile) * kTile;
  const int64_t qa = p->q_tile_pos[static_cast<size_t>(qr) * p->n_qt + qt];
  const int64_t ka = p->kv_tile_pos[static_cast<size_t>(kr) * p->n_kt + kt];
  const int64_t kb = ka + kTile - 1;
  int64_t n = 0;
  for (int i = 0; i < kTile; ++i) {
    const int64_t q = qa + i;
    const int64_t lo = std::max(ka, row_lo_host(p, q));
    const int64_t hi = std::min(kb, q);
    if (hi >= lo) n += hi - lo + 1;
  }
  return n;
}

cp_attn_status build_plan(cp_attn_plan_s* p, const cp_attn_plan_desc* desc) {
  if (!desc) return fail(CP_ATTN_ERR_INVALID_ARG, "plan: null descriptor");
  const int64_t N = desc->seq_len, P = desc->kv_prefix_len;
  const int R = desc->cp;
  if (N <= 0 || P < 0 || R < 1)
    return fail(CP_ATTN_ERR_SHAPE, "plan: need seq_len > 0, kv_prefix_len >= 0, cp >= 1");
  if (desc->n_q_heads <= 0 || desc->n_kv_heads <= 0 || desc->n_q_heads % desc->n_kv_heads)
    return fail(CP_ATTN_ERR_SHAPE, "plan: n_q_heads must be a positive multiple of n_kv_heads");
  if (desc->head_dim != 64 && desc->head_dim != 128)
    return fail(CP_ATTN_ERR_UNSUPPORTED, "plan: head_dim must be 64 or 128");
  if (desc->layout != CP_ATTN_LAYOUT_ZIGZAG && desc->layout != CP_ATTN_LAYOUT_CONTIGUOUS &&
      desc->layout != CP_ATTN_LAYOUT_USP)
    return fail(CP_ATTN_ERR_INVALID_ARG, "plan: unknown layout");
  const int a2a = desc->layout == CP_ATTN_LAYOUT_USP ? desc->a2a : 1;
  if (a2a < 1) return fail(CP_ATTN_ERR_SHAPE, "plan: a2a must be >= 1");
  if (desc->variant != CP_ATTN_PASS_KV && desc->variant != CP_ATTN_PASS_Q &&
      desc->variant != CP_ATTN_VARIANT_AUTO)
    return fail(CP_ATTN_ERR_INVALID_ARG, "plan: unknown variant");
  if (desc->window < 0) return fail(CP_ATTN_ERR_SHAPE, "plan: window must be >= 0");
  const int64_t unit = (desc->layout == CP_ATTN_LAYOUT_CONTIGUOUS ? 1LL * R : 2LL * R * a2a) * kTile;
  if (N % unit != 0 || P % unit != 0)
    return fail(CP_ATTN_ERR_SHAPE,
                "plan: seq_len and kv_prefix_len must be multiples of " +
                    std::to_string(unit) + " (every chunk a multiple of 128 tokens)");
  if (desc->batch < 0) return fail(CP_ATTN_ERR_SHAPE, "plan: batch must be >= 0");
  const int64_t B = desc->batch > 0 ? desc->batch : 1;
  if (B * (N + P) > (1LL << 31) - 1024)
    return fail(CP_ATTN_ERR_SHAPE, "plan: total tokens must fit in int32 positions");
  if (!(desc->softmax_scale >= 0.f) || std::isinf(desc->softmax_scale))
    return fail(CP_ATTN_ERR_INVALID_ARG, "plan: softmax_scale must be finite and >= 0");
  for (cp_attn_dtype t : {desc->partial_dtype, desc->grad_dtype})
    if (t != CP_ATTN_F32 && t != CP_ATTN_BF16)
      return fail(CP_ATTN_ERR_INVALID_ARG, "plan: partial_dtype and grad_dtype must be F32 or BF16");

  p->N = N;
  p->P = P;
  p->B = B;
  p->R = R;
  p->Hq = desc->n_q_heads;
  p->Hkv = desc->n_kv_heads;
  p->d = desc->head_dim;
  p->layout = desc->layout;
  p->a2a = a2a;
  p->part_bf16 = desc->partial_dtype == CP_ATTN_BF16 ? 1 : 0;
  p->grad_bf16 = desc->grad_dtype == CP_ATTN_BF16 ? 1 : 0;
  p->variant = desc->variant == CP_ATTN_VARIANT_AUTO
                   ? select_variant_rule(N, P, desc->n_q_heads, desc->n_kv_heads)
                   : desc->variant;
  // a window as long as a whole sequence masks nothing
  p->window = desc->window >= N + P ? 0 : desc->window;
  p->scale = desc->softmax_scale > 0.f ? desc->softmax_scale
                                       : static_cast<float>(1.0 / std::sqrt(static_cast<double>(p->d)));
  // documents; sequence b of the batch occupies positions [b L, (b + 1) L)
  p->cu.clear();
  const int64_t L = N + P;
  const int64_t total = B * L;
  if (desc->cu_seqlens) {
    if (desc->n_docs < 1) return fail(CP_ATTN_ERR_SHAPE, "plan: n_docs must be >= 1");
    for (int i = 0; i <= desc->n_docs; ++i) p->cu.push_back(desc->cu_seqlens[i]);
    if (p->cu.front() != 0 || p->cu.back() != total)
      return fail(CP_ATTN_ERR_SHAPE,
                  "plan: cu_seqlens must start at 0 and end at batch * (kv_prefix_len + seq_len)");
    for (int i = 0; i < desc->n_docs; ++i)
      if (p->cu[i + 1] <= p->cu[i])
        return fail(CP_ATTN_ERR_SHAPE, "plan: cu_seqlens must be strictly increasing");
    for (int64_t b = 1; b < B; ++b)
      if (!std::binary_search(p->cu.begin(), p->cu.end(), static_cast<int32_t>(b * L)))
        return fail(CP_ATTN_ERR_SHAPE, "plan: cu_seqlens must contain every sequence start");
  } else {
    for (int64_t b = 0; b <= B; ++b) p->cu.push_back(static_cast<int32_t>(b * L));
  }

  // positions: per rank, its shard of sequence 0, then of sequence 1, ...
  p->n_q = B * N / R;
  p->n_kv = B * L / R;
  p->T_q = B * N;
  p->T_kv = B * L;
  p->n_qt = static_cast<int>(p->n_q / kTile);
  p->n_kt = static_cast<int>(p->n_kv / kTile);
  p->q_pos.clear();
  p->kv_pos.clear();
  for (int r = 0; r < R; ++r)
    for (int64_t b = 0; b < B; ++b) shard(N, R, p->layout, p->a2a, b * L + P, r, p->q_pos);
  for (int r = 0; r < R; ++r)
    for (int64_t b = 0; b < B; ++b) {
      if (P > 0) shard(P, R, p->layout, p->a2a, b * L, r, p->kv_pos);
      shard(N, R, p->layout, p->a2a, b * L + P, r, p->kv_pos);
    }
  p->q_tile_pos.resize(static_cast<size_t>(R) * p->n_qt);
  p->kv_tile_pos.resize(static_cast<size_t>(R) * p->n_kt);
  for (size_t i = 0; i < p->q_tile_pos.size(); ++i) {
    p->q_tile_pos[i] = static_cast<int32_t>(p->q_pos[i * kTile]);
    if (p->q_pos[i * kTile + kTile - 1] != p->q_pos[i * kTile] + kTile - 1)
      return fail(CP_ATTN_ERR_SHAPE, "plan: internal error, query tile not contiguous");
  }
  for (size_t i = 0; i < p->kv_tile_pos.size(); ++i) {
    p->kv_tile_pos[i] = static_cast<int32_t>(p->kv_pos[i * kTile]);
    if (p->kv_pos[i * kTile + kTile - 1] != p->kv_pos[i * kTile] + kTile - 1)
      return fail(CP_ATTN_ERR_SHAPE, "plan: internal error, key tile not contiguous");
  }

  // schedule
  p->sched.assign(static_cast<size_t>(R) * R * 2, 0);
  for (int t = 0; t < R; ++t)
    for (int r = 0; r < R; ++r) {
      const int other = ((r - t) % R + R) % R;
      const int qo = p->variant == CP_ATTN_PASS_KV ? r : other;
      const int ko = p->variant == CP_ATTN_PASS_KV ? other : r;
      p->sched[(static_cast<size_t>(t) * R + r) * 2 + 0] = qo;
      p->sched[(static_cast<size_t>(t) * R + r) * 2 + 1] = ko;
    }

  // work lists
  p->fwd_items.clear();
  p->bwd_items.clear();
  p->fwd_off.assign(R + 1, 0);
  p->fwd_nonempty.assign(R, 0);
  p->bwd_off.assign(R + 1, 0);
  p->step_pairs.assign(R, 0);
  auto by_cost = [](const WorkItem& a, const WorkItem& b) {
    return (a.hi - a.lo) > (b.hi - b.lo);
  };
  std::vector<int> cls(static_cast<size_t>(p->n_qt) * p->n_kt);
  // A rank's rows are sequence-major: q tiles [b sq, (b + 1) sq) and kv tiles
  // [b sk, (b + 1) sk) belong to sequence b, and tiles of different sequences
  // are EMPTY, so only a sequence's own tiles are classified.
  const int sq = static_cast<int>(p->n_qt / B), sk = static_cast<int>(p->n_kt / B);
  for (int t = 0; t < R; ++t) {
    std::vector<WorkItem> fwd, bwd;
    for (int r = 0; r < R; ++r) {
      const int qo = p->sched[(static_cast<size_t>(t) * R + r) * 2 + 0];
      const int ko = p->sched[(static_cast<size_t>(t) * R + r) * 2 + 1];
      for (int i = 0; i < p->n_qt; ++i) {
        const int j0 = (i / sq) * sk;
        for (int j = j0; j < j0 + sk; ++j) {
          const int c = tile_class(p, qo, i, ko, j);
          cls[static_cast<size_t>(i) * p->n_kt + j] = c;
          if (c == 2) p->step_pairs[t] += static_cast<int64_t>(kTile) * kTile;
          else if (c == 1) p->step_pairs[t] += tile_visible_pairs(p, qo, i, ko, j);
        }
      }
      // forward: per q tile, its run of non-empty kv tiles (of its sequence)
      for (int i = 0; i < p->n_qt; ++i) {
        int lo = -1, hi = -1, nfull = 0;
        const int j0 = (i / sq) * sk;
        for (int j = j0; j < j0 + sk; ++j) {
          const int c = cls[static_cast<size_t>(i) * p->n_kt + j];
          if (c) {
            if (lo < 0) lo = j;
            else if (hi != j) return fail(CP_ATTN_ERR_UNSUPPORTED, "plan: internal error, non-contiguous kv tile run");
            hi = j + 1;
            nfull += (c == 2);
          }
        }
        if (lo < 0) lo = hi = 0;
        fwd.push_back(WorkItem{qo, ko, i, lo, hi, nfull, 0, 0});
      }
      // backward: per kv tile, its run of non-empty q tiles (of its sequence)
      for (int j = 0; j < p->n_kt; ++j) {
        int lo = -1, hi = -1, nfull = 0;
        const int i0 = (j / sk) * sq;
        for (int i = i0; i < i0 + sq; ++i) {
          const int c = cls[static_cast<size_t>(i) * p->n_kt + j];
          if (c) {
            if (lo < 0) lo = i;
            else if (hi != i) return fail(CP_ATTN_ERR_UNSUPPORTED, "plan: internal error, non-contiguous q tile run");
            hi = i + 1;
            nfull += (c == 2);
          }
        }
        if (lo >= 0) bwd.push_back(WorkItem{qo, ko, j, lo, hi, nfull, 0, 0});
      }
    }
    // longest first: heavy tiles start in the first wave
    std::stable_sort(fwd.begin(), fwd.end(), by_cost);
    std::stable_sort(bwd.begin(), bwd.end(), by_cost);
    int nonempty = 0;
    for (const auto& w : fwd) nonempty += (w.hi > w.lo);
    p->fwd_off[t] = static_cast<int>(p->fwd_items.size());
    p->fwd_nonempty[t] = nonempty;
    p->fwd_items.insert(p->fwd_items.end(), fwd.begin(), fwd.end());
    p->bwd_off[t] = static_cast<int>(p->bwd_items.size());
    p->bwd_items.insert(p->bwd_items.end(), bwd.begin(), bwd.end());
  }
  p->fwd_off[R] = static_cast<int>(p->fwd_items.size());
  p->bwd_off[R] = static_cast<int>(p->bwd_items.size());
  return CP_ATTN_OK;
}

}  // namespace cpa
