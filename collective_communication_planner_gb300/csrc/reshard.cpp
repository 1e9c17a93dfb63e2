// M-to-N reshard planner. See reshard.h.
#include "reshard.h"

#include <algorithm>

namespace tccl {

namespace {

uint64_t ceil_div(uint64_t a, uint64_t b) { return (a + b - 1) / b; }

void mesh_coords(const MeshLayout& l, int m, int* c) {
  for (int a = l.ndims - 1; a >= 0; --a) {
    c[a] = m % l.dims[a];
    m /= l.dims[a];
  }
}

bool same_box(const Box& a, const Box& b, int nd) {
  for (int d = 0; d < nd; ++d)
    if (a.lo[d] != b.lo[d] || a.hi[d] != b.hi[d]) return false;
  return true;
}

bool intersect(const Box& a, const Box& b, int nd, Box* x) {
  for (int d = 0; d < nd; ++d) {
    x->lo[d] = std::max(a.lo[d], b.lo[d]);
    x->hi[d] = std::min(a.hi[d], b.hi[d]);
    if (x->lo[d] >= x->hi[d]) return false;
  }
  return true;
}

struct Block {
  Box box;
  std::vector<int> ranks;  // mesh ranks holding this block (replicas)
};

std::vector<Block> blocks_of(const MeshLayout& l, int nd, const uint64_t* shape) {
  std::vector<Block> out;
  for (int m = 0; m < l.size(); ++m) {
    Box b = layout_box(l, nd, shape, m);
    bool found = false;
    for (Block& k : out)
      if (same_box(k.box, b, nd)) {
        k.ranks.push_back(m);
        found = true;
        break;
      }
    if (!found) out.push_back({b, {m}});
  }
  return out;
}

}  // namespace

bool check_layout(const MeshLayout& l, int nd, const uint64_t* shape, std::string* why) {
  if (l.ndims < 1 || l.ndims > kMaxMeshDims) {
    *why = "a mesh has 1 to 4 dimensions";
    return false;
  }
  int sharded = 0;
  for (int a = 0; a < l.ndims; ++a) {
    if (l.dims[a] < 1) {
      *why = "mesh dimensions must be positive";
      return false;
    }
    const int d = l.place[a];
    if (d == kReplicate) continue;
    if (d < 0 || d >= nd) {
      *why = "a placement shards a dimension the tensor does not have";
      return false;
    }
    if (shape[d] % (uint64_t)l.dims[a]) {
      *why = "a sharded tensor dimension must divide evenly over its mesh axis";
      return false;
    }
    ++sharded;
  }
  if (sharded > 1) {
    *why = "at most one sharded mesh axis per layout";
    return false;
  }
  if (l.size() > kMaxRanks || l.start < 0) {
    *why = "a mesh holds 1 to 64 ranks from a non-negative base rank";
    return false;
  }
  return true;
}

Box layout_box(const MeshLayout& l, int nd, const uint64_t* shape, int m) {
  Box b;
  for (int d = 0; d < nd; ++d) {
    b.lo[d] = 0;
    b.hi[d] = shape[d];
  }
  int c[kMaxMeshDims];
  mesh_coords(l, m, c);
  for (int a = 0; a < l.ndims; ++a) {
    const int d = l.place[a];
    if (d == kReplicate) continue;
    const uint64_t step = shape[d] / (uint64_t)l.dims[a];
    b.lo[d] = (uint64_t)c[a] * step;
    b.hi[d] = b.lo[d] + step;
  }
  return b;
}

bool plan_reshard(const MeshLayout& src, const MeshLayout& dst, int nd, const uint64_t* shape,
                  int es, const uint8_t* src_mod16, const uint8_t* dst_mod16, int sm_count,
                  int cta_cap, int engine, size_t smem_per_block, ReshardPlan* out,
                  std::string* why) {
  *out = ReshardPlan();
  if (nd < 1 || nd > kMaxTensorDims) {
    *why = "a tensor has 1 to 4 dimensions";
    return false;
  }
  for (int d = 0; d < nd; ++d)
    if (shape[d] == 0) {
      *why = "empty tensor dimension";
      return false;
    }
  if (!check_layout(src, nd, shape, why) || !check_layout(dst, nd, shape, why)) return false;
  // the article's constraint: the two meshes are disjoint sets of ranks
  if (src.start < dst.start + dst.size() && dst.start < src.start + src.size()) {
    *why = "source and destination meshes must not share ranks";
    return false;
  }
  const std::vector<Block> sb = blocks_of(src, nd, shape);
  const std::vector<Block> db = blocks_of(dst, nd, shape);
  out->src_load.assign(src.size(), 0);

  // interval intersection; each piece read once from the least-loaded replica
  for (const Block& B : db) {
    uint64_t mask = 0;
    for (int r : B.ranks) mask |= 1ull << r;
    for (const Block& A : sb) {
      Box x;
      if (!intersect(A.box, B.box, nd, &x)) continue;
      int best = A.ranks[0];
      for (int r : A.ranks)
        if (out->src_load[r] < out->src_load[best]) best = r;
      out->src_load[best]++;
      out->transfers.push_back({best, mask, x});
    }
  }

  // lowering: every transfer becomes strided row copies in local buffers
  for (const ReshardTransfer& t : out->transfers) {
    const Box A = layout_box(src, nd, shape, t.src_rank);
    int first_dst = 0;
    while (!((t.dst_mask >> first_dst) & 1ull)) ++first_dst;
    const Box B = layout_box(dst, nd, shape, first_dst);
    uint64_t xe[kMaxTensorDims], ae[kMaxTensorDims], be[kMaxTensorDims];
    uint64_t as[kMaxTensorDims], bs[kMaxTensorDims];  // row-major element strides
    for (int d = 0; d < nd; ++d) {
      xe[d] = t.box.hi[d] - t.box.lo[d];
      ae[d] = A.hi[d] - A.lo[d];
      be[d] = B.hi[d] - B.lo[d];
    }
    as[nd - 1] = bs[nd - 1] = 1;
    for (int d = nd - 2; d >= 0; --d) {
      as[d] = as[d + 1] * ae[d + 1];
      bs[d] = bs[d + 1] * be[d + 1];
    }
    // the contiguous run: trailing dimensions the piece covers entirely in
    // both local buffers, plus the first one it does not
    int k = nd - 1;
    uint64_t run = xe[k];
    while (k > 0 && xe[k] == ae[k] && xe[k] == be[k]) {
      --k;
      run *= xe[k];
    }
    const int row_dim = k - 1;  // -1: a single row
    const uint64_t nrows = row_dim >= 0 ? xe[row_dim] : 1;
    // dimensions outside the row dimension: one window per combination
    uint64_t outer = 1;
    for (int d = 0; d < row_dim; ++d) outer *= xe[d];
    for (uint64_t o = 0; o < outer; ++o) {
      uint64_t idx[kMaxTensorDims] = {0, 0, 0, 0};
      uint64_t rem = o;
      for (int d = row_dim - 1; d >= 0; --d) {
        idx[d] = rem % xe[d];
        rem /= xe[d];
      }
      uint64_t so = 0, dof = 0;
      for (int d = 0; d < nd; ++d) {
        const uint64_t g = t.box.lo[d] + (d < row_dim ? idx[d] : 0);
        so += (g - A.lo[d]) * as[d];
        dof += (g - B.lo[d]) * bs[d];
      }
      ReshardWindow w{};
      w.src_off = so * es;
      w.dst_off = dof * es;
      w.src_pitch = row_dim >= 0 ? as[row_dim] * es : 0;
      w.dst_pitch = row_dim >= 0 ? bs[row_dim] * es : 0;
      w.dst_mask = t.dst_mask;
      w.bytes = (uint32_t)(run * es);
      w.nrows = (uint32_t)nrows;
      w.src = (uint32_t)t.src_rank;
      bool vec = w.bytes % 16 == 0 && (src_mod16[t.src_rank] + w.src_off) % 16 == 0 &&
                 (nrows == 1 || (w.src_pitch % 16 == 0 && w.dst_pitch % 16 == 0));
      for (int r = 0; r < dst.size() && vec; ++r)
        if (((t.dst_mask >> r) & 1ull) && (dst_mod16[r] + w.dst_off) % 16 != 0) vec = false;
      w.scalar = vec ? 0 : 1;
      if (run * es > 0xFFFFFFFFull || nrows > 0xFFFFFFFFull) {
        *why = "a reshard row is too long";
        return false;
      }
      out->win.push_back(w);
      out->bytes_read += run * es * nrows;
      out->bytes_written += run * es * nrows * (uint64_t)__builtin_popcountll(t.dst_mask);
    }
  }
  // the bulk engine takes a plan whose every window is 16-byte co-aligned
  // (whole-vector rows and pitches); one element-wise window sends the whole
  // plan to the warps. Under Auto it also wants a high fan-out and long rows:
  // GB300, 8192 x 8192 bf16 (bulk ring vs warp copies, share of HBM peak):
  // 8 replicas 0.998 vs 0.893, 4 replicas 0.953 vs 0.889, 2 replicas 0.894 vs
  // 0.926, and 2 KiB rows (one thread issues every copy) 0.40 vs 0.93.
  const size_t ring = kReshardBulkHeadBytes + (size_t)kReshardBulkStages * kReshardBulkSegBytes;
  bool bulk = engine != kEngineWarp && engine != kEngineVec && !out->win.empty() &&
              ring <= smem_per_block;
  for (const ReshardWindow& w : out->win) bulk = bulk && !w.scalar;
  if (bulk && engine != kEngineBulk) {
    bulk = out->bytes_written >= kReshardBulkMinFanout * out->bytes_read;
    for (const ReshardWindow& w : out->win) bulk = bulk && w.bytes >= kReshardBulkMinRowBytes;
  }
  out->engine = bulk ? kReshardBulk : kReshardWarp;
  out->unit_prefix.assign(out->win.size() + 1, 0);
  for (size_t i = 0; i < out->win.size(); ++i) {
    const ReshardWindow& w = out->win[i];
    uint64_t units;
    if (bulk) units = bulk_units(w.bytes, w.nrows);
    else if (w.scalar) units = ceil_div(w.bytes / es, kReshardSegElems) * w.nrows;
    else units = ceil_div(w.bytes, kReshardSegBytes) * w.nrows;
    out->unit_prefix[i + 1] = out->unit_prefix[i] + units;
  }
  const uint64_t units = out->unit_prefix.back();
  if (bulk) {
    // one CTA per SM: its ring holds 128 KiB in flight
    uint64_t cap = (uint64_t)std::max(1, sm_count);
    if (cta_cap > 0) cap = std::min<uint64_t>(cap, (uint64_t)cta_cap);
    out->grid = (int)std::max<uint64_t>(1, std::min(units, cap));
    out->threads = kReshardBulkThreads;
    out->smem = ring;
  } else {
    uint64_t blocks = std::max<uint64_t>(1, ceil_div(units, 8));  // 8 warps per CTA
    uint64_t cap = (uint64_t)std::max(1, sm_count) * 8;
    if (cta_cap > 0) cap = std::min<uint64_t>(cap, (uint64_t)cta_cap);
    out->grid = (int)std::min(blocks, cap);
    out->threads = 256;
    out->smem = 0;
  }
  return true;
}

}  // namespace tccl
