// Task planner and lowering pass. See plan.h.
#include "plan.h"

#include <algorithm>
#include <cstdio>
#include <cstring>

namespace tccl {

namespace {

uint64_t ceil_div(uint64_t a, uint64_t b) { return (a + b - 1) / b; }
uint64_t round_up(uint64_t a, uint64_t m) { return ceil_div(a, m) * m; }

constexpr uint32_t kMaxWindowBytes = 1u << 30;

struct PhysTask {
  int src_sel;
  int dst_sel;
  uint64_t src_off;
  uint64_t dst_off;
  uint64_t bytes;
  int task;
};

std::vector<Interval> all_ranks(int p, uint64_t b, uint64_t e) {
  std::vector<Interval> v;
  v.reserve(p);
  for (int r = 0; r < p; ++r) v.push_back({r, b, e});
  return v;
}

// A task's interval list selects either every rank at one common interval
// (sel = -1) or a single rank (sel = that rank).
bool selection(const std::vector<Interval>& iv, int p, int es, int* sel, uint64_t* off,
               uint64_t* bytes) {
  if (iv.empty()) return false;
  for (const Interval& x : iv)
    if (x.begin != iv[0].begin || x.end != iv[0].end) return false;
  if ((int)iv.size() == p && p > 1) {
    for (int r = 0; r < p; ++r)
      if (iv[r].rank != r) return false;
    *sel = -1;
  } else if (iv.size() == 1) {
    *sel = (p == 1) ? -1 : iv[0].rank;
  } else {
    return false;
  }
  *off = iv[0].begin * (uint64_t)es;
  *bytes = (iv[0].end - iv[0].begin) * (uint64_t)es;
  return true;
}

// Merges neighbours that continue each other (same selections, adjacent
// offsets, both 16-byte bodies): for allreduce this folds the P shard bodies
// into one window.
std::vector<Window> merge_adjacent(const std::vector<Window>& wins) {
  std::vector<Window> m;
  for (const Window& w : wins) {
    if (!m.empty()) {
      Window& b = m.back();
      if (!b.scalar && !w.scalar && b.src_sel == w.src_sel && b.dst_sel == w.dst_sel &&
          b.src_off + b.bytes == w.src_off && b.dst_off + b.bytes == w.dst_off &&
          (uint64_t)b.bytes + w.bytes <= 0xFFFFFFF0ull) {
        b.bytes += w.bytes;
        continue;
      }
    }
    m.push_back(w);
  }
  return m;
}

void push_split(std::vector<Window>& out, Window w, uint64_t bytes, uint32_t limit) {
  while (bytes > 0) {
    uint64_t n = std::min<uint64_t>(bytes, limit);
    w.bytes = (uint32_t)n;
    out.push_back(w);
    w.src_off += n;
    w.dst_off += n;
    bytes -= n;
  }
}

}  // namespace

uint64_t message_bytes(int coll, int nranks, uint64_t count, int elem_size) {
  if (coll == kAllReduce) return count * (uint64_t)elem_size;
  return (uint64_t)nranks * count * (uint64_t)elem_size;
}

Plan plan_collective(int coll, int nranks, uint64_t count, int elem_size, int op) {
  Plan pl;
  pl.coll = coll;
  pl.nranks = nranks;
  pl.elem_size = elem_size;
  pl.op = op;
  pl.count = count;
  const int p = nranks;
  if (coll == kAllReduce) {
    // shard length: ceil(count / P), rounded up so every shard starts 16-byte
    // aligned relative to the buffer base; trailing shards may be short or empty
    uint64_t q = round_up(ceil_div(count, (uint64_t)p), 16 / (uint64_t)elem_size);
    pl.shard_elems = q;
    for (int s = 0; s < p; ++s) {
      uint64_t b = std::min<uint64_t>((uint64_t)s * q, count);
      uint64_t e = std::min<uint64_t>((uint64_t)(s + 1) * q, count);
      if (b == e) continue;
      LogicalTask in{kShardIn, op, s, s, kSendBuf, kOwnerShard, all_ranks(p, b, e), {{s, b, e}},
                     {}};
      int in_idx = (int)pl.tasks.size();
      pl.tasks.push_back(in);
      LogicalTask out{kShardOut, -1, s, s, kOwnerShard, kRecvBuf, {{s, b, e}}, all_ranks(p, b, e),
                      {in_idx}};
      pl.tasks.push_back(out);
    }
  } else if (coll == kReduceScatter) {
    pl.shard_elems = count;
    if (count == 0) return pl;
    for (int s = 0; s < p; ++s) {
      uint64_t b = (uint64_t)s * count, e = b + count;
      pl.tasks.push_back({kShardIn, op, s, s, kSendBuf, kRecvBuf, all_ranks(p, b, e),
                          {{s, 0, count}}, {}});
    }
  } else {
    pl.shard_elems = count;
    if (count == 0) return pl;
    for (int s = 0; s < p; ++s) {
      uint64_t b = (uint64_t)s * count, e = b + count;
      pl.tasks.push_back({kShardOut, -1, s, s, kSendBuf, kRecvBuf, {{s, 0, count}},
                          all_ranks(p, b, e), {}});
    }
  }
  return pl;
}

uint64_t small_max_bytes(const Config& c, int nranks) {
  // 0: by rank count. Graph-captured on GB300 (the warp engine against the vec
  // engine with its small CTAs spread over the SMs, both with the rank count
  // compiled in): from P = 5 to 8 the vec engine is about as fast at 64 KiB per
  // rank and faster above (P = 8, 128 KiB: 1.6-1.8 against 2.2 us; P = 6:
  // 1.65 against 1.97); at P = 3 and 4 the two tie up to 128 KiB; at P = 16
  // they tie at 16 KiB and the vec engine is faster from 64 KiB (2.4 against
  // 2.7 us).
  if (c.small_max_bytes) return c.small_max_bytes;
  return nranks >= 5 ? 64 * 1024 : 128 * 1024;
}

Config resolve_config(const Config& in) {
  Config c = in;
  // defaults chosen by launch-shape sweeps on GB300 (P = 4 and 8, bf16)
  if (c.vec_max_bytes == 0) c.vec_max_bytes = 4 * 1024 * 1024;
  if (c.stage_bytes <= 0) c.stage_bytes = kDefaultStageBytes;
  if (c.stages <= 0) c.stages = kDefaultStages;
  if (c.consumer_warps <= 0) c.consumer_warps = 16;
  if (c.consumer_warps > kMaxConsumerWarps) c.consumer_warps = kMaxConsumerWarps;
  if (c.stage_layout < kLayoutAuto || c.stage_layout > kLayoutPerRank) c.stage_layout = kLayoutAuto;
  if (c.ctas_per_sm <= 0) c.ctas_per_sm = 1;
  if (c.ctas_per_sm > 4) c.ctas_per_sm = 4;
  if (c.wait_timeout_ms <= 0) c.wait_timeout_ms = 2000.0;
  if (c.chunk_order < kOrderAuto || c.chunk_order > kOrderDynamic) c.chunk_order = kOrderAuto;
  if (c.prefetch_chunks < 0) c.prefetch_chunks = 0;
  if (c.prefetch_chunks > 64) c.prefetch_chunks = 64;
  if (c.load_policy < 0 || c.load_policy > 2) c.load_policy = 0;
  if (c.max_chunk_bytes == 0) c.max_chunk_bytes = kDefaultMaxChunkBytes;
  c.max_chunk_bytes = std::min<size_t>(std::max<size_t>(c.max_chunk_bytes, 256), 65536) & ~(size_t)15;
  // copy engines: four streams and pieces of 16 MiB or more sustained
  // ~4.8 TB/s of fan-out copies in a GB300 probe (one stream ~2.5, 2 MiB
  // pieces ~1.1); segments up to 28 MiB per rank: a 128 MiB-per-rank
  // allreduce (P = 8, bf16) then runs in five segments, the last of 16 MiB,
  // whose copies (which overlap no fold) end sooner: 0.312 / 0.528 / 0.744 /
  // 0.812 of the HBM peak at caps 8 / 16 / 32 / 47 against 0.310 / 0.519 /
  // 0.736 / 0.789 in four of 32 MiB (26 and 30 MiB: at or below 28)
  if (c.ce_streams <= 0) c.ce_streams = 4;
  if (c.ce_streams > 8) c.ce_streams = 8;
  if (c.ce_segment_bytes == 0) c.ce_segment_bytes = (size_t)28 << 20;
  c.ce_segment_bytes = std::min<size_t>(std::max<size_t>(c.ce_segment_bytes, 4096), (size_t)1 << 30) & ~(size_t)255;
  if (c.reduce_order != 1) c.reduce_order = 0;
  if (c.ce_fold < kFoldAuto || c.ce_fold > kFoldTmaReduce) c.ce_fold = kFoldAuto;
  if (c.ce_tail_percent <= 0 || c.ce_tail_percent > 100) c.ce_tail_percent = 100;
  if (c.reduce_slots < 0 || c.reduce_slots > kMaxReduceSlots) c.reduce_slots = 0;
  if (c.ce_ar_streams < 0) c.ce_ar_streams = 0;  // 0: by the cap (copy_out_streams)
  if (c.ce_tail_streams <= 0) c.ce_tail_streams = c.ce_streams;
  c.ce_ar_streams = std::min(c.ce_ar_streams, c.ce_streams);
  c.ce_tail_streams = std::min(c.ce_tail_streams, c.ce_streams);
  return c;
}

int copy_out_auto_max_cap(const Config& c, int sm_count, int nranks) {
  if (c.ce_auto_max_cap > 0) return c.ce_auto_max_cap;
  // allreduce / all-gather: the cap up to which the copy-out engine (its
  // fold with 256-bit loads) stays ahead of the SM-only bulk engine. GB300
  // allreduce, bf16, 128 MiB per rank, share of the HBM peak, copy-out / SM
  // only: P = 2 cap 80 0.705 / 0.664, 96 0.718 / 0.786; P = 3 cap 60
  // 0.729 / 0.690, 64 0.731 / 0.732; P = 4 cap 60 0.800 / 0.780, 64
  // 0.806 / 0.820; P = 5 cap 68 0.816 / 0.809, 72 0.758 / 0.842; P = 8 cap
  // 66 0.859 / 0.846, 68 0.855 / 0.865. (A copy-out all-gather uses no SM
  // and stays ahead further.)
  if (nranks <= 2) return sm_count * 4 / 7;
  if (nranks <= 4) return sm_count * 5 / 12;
  return sm_count * 7 / 16;
}

bool copy_out_chosen(const Config& c, int sm_count, int nranks, int coll, size_t count, int es,
                     int cap) {
  if (nranks < 2) return false;
  if (c.engine == kEngineCopyOut) return true;
  if (c.engine != kEngineAuto || c.ce_auto_max_cap < 0) return false;
  const size_t per_rank = count * (size_t)es * (coll == kAllReduce ? 1 : (size_t)nranks);
  if (per_rank < kCeAutoMinBytes) return false;
  // GB300 sweeps: the reduce-scatter's register fold beats the TMA pipeline
  // under every cap, and uncapped for up to four ranks (0.995 vs 0.959 of
  // the HBM peak at P = 4, 64 MiB; 0.982 vs 1.045 at P = 8)
  if (coll == kReduceScatter) return cap > 0 || nranks <= 4;
  if (cap <= 0) return false;
  return cap <= copy_out_auto_max_cap(c, sm_count, nranks);
}

void copy_out_segments(const Config& c, size_t count, int es, size_t* seg_elems, int* nseg) {
  // the copies of the first segment and the fold of the last one overlap
  // nothing, so segments should be short; but each costs a launch
  const size_t align = 256 / (size_t)es;
  const size_t quarter = std::max<size_t>((size_t)4 << 20, (count * es + 3) / 4);
  const size_t seg_bytes = std::min<size_t>(c.ce_segment_bytes, quarter);
  size_t seg = std::max<size_t>(align, (seg_bytes / (size_t)es) / align * align);
  if ((count + seg - 1) / seg > (size_t)kMaxCeSegments)
    seg = ((count + kMaxCeSegments - 1) / kMaxCeSegments + align - 1) / align * align;
  const size_t n = (count + seg - 1) / seg;
  if (n >= 2 && c.ce_tail_percent > 0 && c.ce_tail_percent < 100) {
    // n - 1 full segments of s and a last one of about f s: s = count / (n - 1 + f)
    const double f = c.ce_tail_percent / 100.0;
    size_t s = (size_t)((double)count / ((double)(n - 1) + f));
    s = (s + align - 1) / align * align;
    if (s >= seg && (n - 1) * s < count) seg = s;
  }
  *seg_elems = seg;
  *nseg = (int)((count + seg - 1) / seg);
}

bool register_fold_ok(int coll, int nranks, const uint8_t* send_mod16, const uint8_t* recv_mod16,
                      size_t count, int es, size_t seg_elems) {
  const uint8_t mod = recv_mod16[0];
  for (int k = 0; k < nranks; ++k) {
    if (send_mod16[k] != mod) return false;
    if (coll == kReduceScatter && recv_mod16[k] != mod) return false;
  }
  if (coll == kReduceScatter) {
    const size_t bytes = count * (size_t)es;
    return bytes % 16 == 0 && bytes / 16 < kFoldMaxVectors;
  }
  return seg_elems * (size_t)es / 16 < kFoldMaxVectors;
}

void copy_out_streams(const Config& c, int nranks, int cap, int* mid, int* tail) {
  // the copies of a segment run beside the next segment's fold, whose length
  // goes as 1 / cap: more copies at once slow that fold down (they share the
  // memory system) more than they gain once the copies keep up with it.
  // GB300, C4 (P = 8, bf16, 128 MiB per rank), share of the HBM peak, one
  // stream for the overlapped segments against two / three / four: cap 8
  // 0.306 / 0.303 / 0.303 / 0.298, cap 16 0.512 / 0.508 / 0.508 / 0.497;
  // cap 32 two or three (0.729-0.733) against one (0.720) and four (0.722).
  // A segment's copies are P - 1 of its size, so the count scales with P - 1
  // as well: one stream per 112 / (P - 1) CTAs, rounded (P = 8: one per 16);
  // P = 4, 64 MiB per rank, cap 32: one stream 0.605, two 0.583.
  int m = c.ce_ar_streams;
  if (m <= 0) m = cap > 0 ? std::max(1, (cap * (nranks - 1) + 56) / 112) : c.ce_streams;
  m = std::min(m, c.ce_streams);
  *mid = std::max(1, std::min(m, nranks - 1));
  *tail = std::max(1, std::min(c.ce_tail_streams, nranks - 1));
}

bool allreduce_register_fold(const Config& c, int nranks, const uint8_t* send_mod16,
                             const uint8_t* recv_mod16, size_t count, int es, size_t seg_elems) {
  if (c.ce_fold == kFoldTma || c.ce_fold == kFoldTmaReduce) return false;
  return register_fold_ok(kAllReduce, nranks, send_mod16, recv_mod16, count, es, seg_elems);
}

// Body windows -> one chunk sequence (prefix table), element-wise windows cut
// into pieces and bound to CTAs, and the grid size. Each CTA runs `lanes`
// independent chunk streams (the TMA-reduce engine) or one (the bulk engine).
void build_chunk_tables(const std::vector<Window>& wins, uint64_t chunk, int lanes,
                        int max_ctas_total, int cta_cap, const Config& cfg, int es, bool capped,
                        Lowered* out) {
  LaunchShape& sh = out->shape;
  std::vector<Window> body, scal;
  uint64_t sbytes = 0;
  for (const Window& w : merge_adjacent(wins)) {
    if (w.scalar) {
      scal.push_back(w);
      sbytes += w.bytes;
    } else {
      body.push_back(w);
    }
  }
  int max_g = max_ctas_total;
  if (cta_cap > 0) max_g = std::min(max_g, cta_cap);
  // body windows -> one sequence of chunks
  out->nbody = (int)body.size();
  out->chunk_prefix.assign(body.size() + 1, 0);
  for (size_t i = 0; i < body.size(); ++i)
    out->chunk_prefix[i + 1] = out->chunk_prefix[i] + ceil_div(body[i].bytes, chunk);
  const uint64_t total = out->chunk_prefix.back();
  out->total_chunks = total;
  int grid = total > 0 ? (int)std::min<uint64_t>(max_g, ceil_div(total, (uint64_t)lanes)) : 1;
  // uncapped: claim chunks dynamically (SMs stream at different rates);
  // capped: a fixed cyclic share per CTA
  int order = cfg.chunk_order != kOrderAuto ? cfg.chunk_order
                                            : (capped ? kOrderCyclic : kOrderDynamic);
  sh.order = order;
  if (total > 0 && order == kOrderBlocked) {
    out->chunks_per_cta = ceil_div(total, (uint64_t)grid);
    grid = (int)ceil_div(total, out->chunks_per_cta);
  }
  // element-wise windows: cut into pieces and bound to CTAs round robin
  std::vector<Window> pieces;
  if (!scal.empty()) {
    uint64_t limit = std::max<uint64_t>(4096, round_up(ceil_div(sbytes, (uint64_t)max_g), es));
    for (const Window& w : scal) {
      Window x = w;
      uint64_t left = w.bytes;
      while (left > 0) {
        uint64_t n = std::min<uint64_t>(left, limit);
        x.bytes = (uint32_t)n;
        pieces.push_back(x);
        x.src_off += n;
        x.dst_off += n;
        left -= n;
      }
    }
    if (total == 0) grid = (int)std::min<uint64_t>(max_g, pieces.size());
    for (size_t i = 0; i < pieces.size(); ++i) pieces[i].cta = (int32_t)(i % (size_t)grid);
    std::stable_sort(pieces.begin(), pieces.end(),
                     [](const Window& x, const Window& y) { return x.cta < y.cta; });
  }
  out->win = body;
  out->win.insert(out->win.end(), pieces.begin(), pieces.end());
  out->cta_first.assign(grid + 1, 0);
  for (const Window& w : pieces) out->cta_first[w.cta + 1]++;
  for (int i = 0; i < grid; ++i) out->cta_first[i + 1] += out->cta_first[i];
  sh.grid = grid;
}

bool lower_plan(const Plan& plan, const uint8_t* send_mod16, const uint8_t* recv_mod16,
                const Config& cfg_in, const DeviceDesc& dev, int cta_cap, Lowered* out,
                std::string* why) {
  const Config cfg = resolve_config(cfg_in);
  const int p = plan.nranks;
  const int es = plan.elem_size;
  *out = Lowered();
  out->ntasks = (int)plan.tasks.size();

  // ---- 1. logical -> physical tasks. A shard-out whose only dependency is
  // the shard-in that produced its source interval is fused with it: the
  // reduced shard then never leaves the chip (loaded once, stored P times).
  std::vector<PhysTask> phys;
  std::vector<char> consumed(plan.tasks.size(), 0);
  for (size_t i = 0; i < plan.tasks.size(); ++i) {
    const LogicalTask& t = plan.tasks[i];
    if (t.kind == kShardOut && t.src_buf == kOwnerShard) {
      if (t.deps.size() != 1) {
        *why = "shard-out with an unexpected dependency list";
        return false;
      }
      const LogicalTask& in = plan.tasks[t.deps[0]];
      if (in.kind != kShardIn || in.dst.size() != 1 || t.src.size() != 1 ||
          in.dst[0].begin != t.src[0].begin || in.dst[0].end != t.src[0].end ||
          in.dst[0].rank != t.src[0].rank) {
        *why = "shard-out does not consume its shard-in's result";
        return false;
      }
      PhysTask pt{};
      uint64_t b1, b2;
      if (!selection(in.src, p, es, &pt.src_sel, &pt.src_off, &b1) ||
          !selection(t.dst, p, es, &pt.dst_sel, &pt.dst_off, &b2) || b1 != b2) {
        *why = "fused shard task has irregular intervals";
        return false;
      }
      pt.bytes = b1;
      pt.task = t.shard;
      consumed[t.deps[0]] = 1;
      phys.push_back(pt);
    }
  }
  for (size_t i = 0; i < plan.tasks.size(); ++i) {
    const LogicalTask& t = plan.tasks[i];
    if (consumed[i] || (t.kind == kShardOut && t.src_buf == kOwnerShard)) continue;
    PhysTask pt{};
    uint64_t b1, b2;
    if (!selection(t.src, p, es, &pt.src_sel, &pt.src_off, &b1) ||
        !selection(t.dst, p, es, &pt.dst_sel, &pt.dst_off, &b2) || b1 != b2) {
      *why = "task has irregular intervals";
      return false;
    }
    pt.bytes = b1;
    pt.task = t.shard;
    phys.push_back(pt);
  }

  // ---- 2. alignment split: a task whose selected source and destination
  // addresses agree mod 16 gets a scalar head, a 16-byte body and a scalar
  // tail; any other task runs element-wise.
  std::vector<Window> wins;
  for (const PhysTask& pt : phys) {
    if (pt.bytes == 0) continue;
    int a = -1;
    bool co = true;
    auto check = [&](int m) {
      if (a < 0) a = m;
      else if (a != m) co = false;
    };
    for (int r = 0; r < p; ++r) {
      if (pt.src_sel < 0 || pt.src_sel == r) check((int)((send_mod16[r] + pt.src_off) & 15));
      if (pt.dst_sel < 0 || pt.dst_sel == r) check((int)((recv_mod16[r] + pt.dst_off) & 15));
    }
    Window w{};
    w.src_sel = (int16_t)pt.src_sel;
    w.dst_sel = (int16_t)pt.dst_sel;
    w.task = (uint16_t)pt.task;
    w.cta = -1;
    w.src_off = pt.src_off;
    w.dst_off = pt.dst_off;
    if (!co) {
      w.scalar = 1;
      push_split(wins, w, pt.bytes, kMaxWindowBytes);
      continue;
    }
    uint64_t head = std::min<uint64_t>(pt.bytes, (uint64_t)((16 - a) & 15));
    uint64_t body = (pt.bytes - head) & ~(uint64_t)15;
    uint64_t tail = pt.bytes - head - body;
    if (head) {
      w.scalar = 1;
      push_split(wins, w, head, kMaxWindowBytes);
      w.src_off += head;
      w.dst_off += head;
    }
    if (body) {
      w.scalar = 0;
      push_split(wins, w, body, kMaxWindowBytes);
      w.src_off += body;
      w.dst_off += body;
    }
    if (tail) {
      w.scalar = 1;
      push_split(wins, w, tail, kMaxWindowBytes);
    }
  }

  // ---- 3. engine choice: the warp engine for the smallest messages (one
  // lane per vector and rank), the vec engine for mid sizes, the bulk (TMA)
  // pipeline for large messages and for every capped large call
  const int max_ctas_total = std::max(1, dev.sm_count) * std::max(1, cfg.ctas_per_sm);
  const bool capped = cta_cap > 0 && cta_cap < max_ctas_total;
  int engine = cfg.engine;
  if (engine == kEngineAuto) {
    const uint64_t mb = message_bytes(plan.coll, p, plan.count, es);
    // an out-of-place allreduce over 8 ranks goes to the vec engine at every
    // small size: graph-captured on GB300, 4-64 KiB per rank, 1.56-1.76 against
    // 1.67-1.86 us on the warp engine (bf16, 16 KiB: 1.66 against 1.80). In
    // place the warp engine stays ahead below 64 KiB (16 KiB: 1.85 against
    // 1.95), and at other rank counts the two were within noise or mixed.
    const bool vec_first = cfg.small_max_bytes == 0 && plan.coll == kAllReduce && !plan.in_place && p == 8;
    if (mb <= small_max_bytes(cfg, p) && !vec_first) engine = kEngineWarp;
    else if (mb <= cfg.vec_max_bytes && !capped) engine = kEngineVec;
    else engine = kEngineBulk;
  }
  // the copy-out engine's kernels are bulk-engine kernels (its copies are
  // issued by the host); a reduce-scatter has nothing to copy out
  if (engine == kEngineCopyOut) engine = kEngineBulk;
  if (engine == kEngineWarp && p > 32) engine = kEngineVec;
  LaunchShape& sh = out->shape;
  sh.engine = engine;

  if (engine == kEngineWarp || engine == kEngineVec) {
    std::vector<Window> m = merge_adjacent(wins);
    out->win = m;
    out->size_class = (p <= kSmallRanks && (int)m.size() <= kSmallWindows) ? 0 : 1;
    if ((int)m.size() > kLargeWindows) {
      *why = "too many windows for the small-message engines";
      return false;
    }
    out->vec_prefix.assign(m.size() + 1, 0);
    out->elem_prefix.assign(m.size() + 1, 0);
    for (size_t i = 0; i < m.size(); ++i) {
      out->vec_prefix[i + 1] = out->vec_prefix[i] + (m[i].scalar ? 0 : m[i].bytes / 16);
      out->elem_prefix[i + 1] = out->elem_prefix[i] + (m[i].scalar ? m[i].bytes / es : 0);
    }
    uint64_t nvec = out->vec_prefix.back();
    uint64_t nelem = out->elem_prefix.back();
    uint64_t lanes;
    if (engine == kEngineWarp) {
      int vpw = 32 / p;  // vectors per warp: one group of P lanes per vector
      lanes = ceil_div(nvec, (uint64_t)vpw) * 32;
    } else {
      lanes = nvec;
    }
    lanes = std::max<uint64_t>(lanes, nelem);
    // the vec engine with few lanes: one CTA per SM, each of the lanes / SMs
    // rounded up to a warp, so that every SM gets the same few lanes. Graph-
    // captured on GB300 (P = 2, 4, 8, f32 and bf16, 16 KiB to 1 MiB per rank,
    // in place and out of place), against fixed CTAs of 128 lanes: 1.75 against
    // 2.1 us at P = 8, 128 KiB in place (64 CTAs on 152 SMs), and no slower
    // beyond noise anywhere up to 192 lanes per SM (P = 8: 384 KiB). From
    // 512 KiB on, CTAs of 256.
    int threads = 256;
    const uint64_t sms = (uint64_t)std::max(1, dev.sm_count);
    if (engine == kEngineVec && lanes <= sms * kVecSpreadLanesPerSm)
      threads = (int)std::max<uint64_t>(32, ceil_div(ceil_div(lanes, sms), (uint64_t)32) * 32);
    uint64_t blocks = std::max<uint64_t>(1, ceil_div(lanes, threads));
    uint64_t cap = (uint64_t)dev.sm_count * 8;
    if (cta_cap > 0) cap = std::min<uint64_t>(cap, (uint64_t)cta_cap);
    sh.grid = (int)std::max<uint64_t>(1, std::min(blocks, cap));
    sh.threads = threads;
    sh.smem = 0;
    sh.early_launch = capped ? 0 : 1;
    return true;
  }

  int smem_budget = dev.smem_optin;
  if (dev.smem_per_sm > 0)
    smem_budget = std::min(smem_budget, dev.smem_per_sm / std::max(1, cfg.ctas_per_sm) - 1024);

  // ---- 4a. TMA-reduce engine: the copy hardware applies the reduction
  if (engine == kEngineTmaReduce) {
    if (plan.coll == kAllGather) {
      *why = "an all-gather has nothing for the TMA-reduce engine to reduce";
      return false;
    }
    // each issuing thread (lane 0 of a warp) keeps `slots` chunks in flight,
    // each double-buffered over the ranks; a reduce-scatter's slots get a
    // third buffer for an in-place owner's own chunk
    const int bufs = plan.coll == kReduceScatter ? 3 : 2;
    int slots = cfg.reduce_slots > 0 ? cfg.reduce_slots : kDefaultReduceSlots;
    uint64_t chunk = cfg.max_chunk_bytes == kDefaultMaxChunkBytes ? kDefaultReduceChunkBytes
                                                                   : (uint64_t)cfg.max_chunk_bytes;
    int lanes = 0;
    for (;;) {
      const int64_t room = (int64_t)smem_budget - 1024;
      lanes = (int)std::min<int64_t>(cfg.consumer_warps, room / (int64_t)(slots * bufs * chunk));
      lanes = std::min(lanes, kReduceMaxBarriers / (slots * bufs));
      if (lanes >= 1) break;
      if (slots > 1) slots /= 2;
      else if (chunk > 1024) chunk = (chunk / 2) & ~(uint64_t)15;
      else break;
    }
    if (lanes < 1) {
      *why = "shared memory too small for the TMA-reduce engine";
      return false;
    }
    sh.chunk_bytes = (int)chunk;
    sh.stages = slots;
    sh.reduce_slots = slots;
    sh.reduce_bufs = bufs;
    sh.consumer_warps = lanes;
    sh.threads = 32 * lanes;
    sh.store_mode = kStoreBulk;
    sh.smem = 1024 + (size_t)lanes * slots * bufs * chunk;
    build_chunk_tables(wins, chunk, lanes * slots, max_ctas_total, cta_cap, cfg, es, capped, out);
    sh.order = kOrderCyclic;  // every (grid x lanes)-th chunk per lane
    return true;
  }

  // ---- 4b. bulk engine: chunks, stages, CTAs
  int layout = cfg.stage_layout;
  if (plan.coll == kAllGather) layout = kLayoutShared;  // one source: nothing to stream
  // many ranks make the shared layout's per-rank copies tiny (64 KiB / P);
  // below 2 KiB per copy the per-rank layout, with whole-stage copies, wins
  if (layout == kLayoutAuto)
    layout = ((uint64_t)cfg.stage_bytes / (uint64_t)p < 2048) ? kLayoutPerRank : kLayoutShared;
  sh.rank_streamed = layout == kLayoutPerRank ? 1 : 0;
  const int nsrc = (plan.coll == kAllGather || sh.rank_streamed) ? 1 : p;
  // all-gather stores straight from the stage; a reduced chunk goes out as
  // bulk stores from a result slot when every SM streams, and as register
  // stores (no extra shared-memory pass) when a cap concentrates the work
  int store = cfg.store_mode;
  if (store == kStoreAuto)
    store = (plan.coll == kAllGather || !capped) ? kStoreBulk : kStoreVec;
  if (sh.rank_streamed) store = kStoreVec;  // the sums leave from registers
  sh.store_mode = store;
  uint64_t chunk = ((uint64_t)cfg.stage_bytes / nsrc) & ~(uint64_t)15;
  chunk = std::min<uint64_t>(chunk, cfg.max_chunk_bytes);
  chunk = std::max<uint64_t>(chunk, 256);
  if (sh.rank_streamed)  // every consumer thread owns kPerRankVectors vectors of a chunk
    chunk = (uint64_t)16 * kPerRankVectors * 32 * cfg.consumer_warps;
  const int result_slots = (store == kStoreBulk && plan.coll != kAllGather) ? 2 : 0;
  const int budget = smem_budget;
  int max_stages = cfg.stages;
  const uint64_t traffic = 2ull * (uint64_t)p * plan.count * (uint64_t)es;
  if (plan.coll == kAllReduce && !plan.in_place && !plan.anchor_only && !capped &&
      !sh.rank_streamed && default_bulk_shape(cfg) && traffic >= kArInflightMinTraffic) {
    // a large out-of-place allreduce streamed best with about 96 KiB of
    // loads in flight per SM, not the most that fits: GB300 sweeps, P = 2 /
    // 4 / 8 / 16 moving 512 MiB - 2 GiB, 0.5-1% faster than 192 KiB (its P
    // stores per chunk keep the other half of the traffic moving). Calls
    // that store once per P loads (a reduce-scatter lost 17% this way), in
    // place (0.5% slower) or smaller (at 256 MiB the two were within 1.5%
    // either way; at 64-128 MiB the full ring was 5-20% faster for P = 4
    // and 8) keep the full ring. Chunks stay at 6 KiB or more: smaller ones
    // cost more per byte than they save. Two stages of 48 KiB where the
    // chunk allows (P=4: 12 KiB chunks, 1.008 of peak at 64 MiB per rank
    // against 0.999 for three stages of 8 KiB, with the first chunks
    // prefetched into L2).
    chunk = std::max<uint64_t>(kArMinChunkBytes,
                               std::min<uint64_t>(cfg.max_chunk_bytes, kArInflightBytes / 2 / nsrc));
    chunk &= ~(uint64_t)15;
    max_stages = (int)std::max<uint64_t>(2, std::min<uint64_t>(cfg.stages, kArInflightBytes / (nsrc * chunk)));
  }
  int stages = 0;
  for (;;) {
    int64_t room = (int64_t)budget - 1024 - (int64_t)result_slots * (int64_t)chunk;
    stages = room > 0 ? (int)std::min<int64_t>(max_stages, room / (int64_t)(nsrc * chunk)) : 0;
    if (stages >= 2 || chunk <= 16 || sh.rank_streamed) break;
    chunk = std::max<uint64_t>(16, (chunk / 2) & ~(uint64_t)15);
  }
  if (stages < 2) {
    *why = "shared memory too small for a two-stage pipeline";
    return false;
  }
  stages = std::min(stages, 32);
  sh.stages = stages;
  sh.chunk_bytes = (int)chunk;
  sh.consumer_warps = cfg.consumer_warps;
  sh.threads = 32 * (1 + cfg.consumer_warps);
  // all-gather bulk stores: keep up to stages - 2 store groups in flight
  // (two stages left for loads); GB300 sweep: P = 4, 64 MiB: 0.928 of the
  // HBM peak against 0.918 with stages / 2, and 0.74 with stages - 1
  sh.release_lag = std::max(1, std::min(7, stages - 2));
  sh.prefetch_chunks = cfg.prefetch_chunks;
  sh.load_evict_first = cfg.load_policy == 1 ? 1 : 0;
  // an uncapped launch may start behind the previous kernel on the stream
  // (its CTAs wait before touching global memory); a capped one never holds
  // SMs beyond its cap
  sh.early_launch = capped ? 0 : 1;
  sh.smem = 1024 + (size_t)stages * nsrc * chunk + (size_t)result_slots * chunk;

  build_chunk_tables(wins, chunk, 1, max_ctas_total, cta_cap, cfg, es, capped, out);
  return true;
}

void pack_bulk_table(const Lowered& low, std::vector<unsigned char>* out, size_t* off_prefix,
                     size_t* off_cta, size_t* off_sched) {
  const size_t wbytes = low.win.size() * sizeof(Window);
  const size_t pbytes = low.chunk_prefix.size() * sizeof(uint64_t);
  const size_t cbytes = low.cta_first.size() * sizeof(uint32_t);
  *off_prefix = wbytes;
  *off_cta = wbytes + pbytes;
  *off_sched = (wbytes + pbytes + cbytes + 15) & ~(size_t)15;  // two zeroed 8-byte words
  out->assign(*off_sched + 16, 0);
  if (wbytes) std::memcpy(out->data(), low.win.data(), wbytes);
  if (pbytes) std::memcpy(out->data() + *off_prefix, low.chunk_prefix.data(), pbytes);
  if (cbytes) std::memcpy(out->data() + *off_cta, low.cta_first.data(), cbytes);
}

}  // namespace tccl
