// Device code for the three engines (sm_103a).
//
// Bulk engine: the T-CCL "TMA engine" ("NCCL M2N vs T-CCL" article, section
// 2.3 and the kernel sketches of section 2.5), rebuilt for one GPU. Each CTA
// is persistent over its windows. One producer thread issues, per chunk, one
// `cp.async.bulk` load per source rank into a shared-memory stage and arms
// the stage's mbarrier with the expected byte count (shard-in load,
// section 2.2 "reduction localisation"). Consumer warps wait on the stage,
// fold the P contributions in ascending rank order in fp32 / int32 registers
// and emit the reduced chunk, which exists once on chip, to every destination
// (section 2.2 "shard-out: load once, reuse for all peer stores"): either as
// P `cp.async.bulk` stores from a shared-memory result slot, or as P 128-bit
// stores from registers. Every wait is bounded; on expiry the kernel records
// a timeout in the group's status word, skips its remaining work and exits.
//
// Warp / vec engines (small messages): no shared memory, no barriers. The
// warp engine gives each (16-byte vector, rank) pair its own lane: lanes load
// one vector each, and every lane of a group of P folds the group's values in
// rank order through warp shuffles, then stores its rank's copy. The vec
// engine gives each vector to one lane, which loads all P contributions.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "internal.h"

namespace tccl {
namespace dev {

// ------------------------------------------------------------------ PTX
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(smem_addr(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// global -> shared bulk copy, completion counted in bytes on `bar`
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// the same, with an L2 cache-eviction policy for the read lines
__device__ __forceinline__ void bulk_load_hint(void* smem_dst, const void* gsrc, uint32_t bytes,
                                               uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// evict-first L2 policy for data read exactly once
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// global -> L2 bulk prefetch (no completion tracking): lets the L2 act as a
// deeper staging level in front of the shared-memory ring
__device__ __forceinline__ void bulk_prefetch_l2(const void* gsrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gsrc), "r"(bytes) : "memory");
}

// shared -> global bulk reduction (element-wise op applied at the destination
// by the memory system), tracked by bulk async-groups like a bulk store
template <int DT, int OP>
__device__ __forceinline__ void bulk_reduce(void* gdst, const void* smem_src, uint32_t bytes) {
  if (DT == kF32) {
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(
                     gdst), "r"(smem_addr(smem_src)), "r"(bytes)
                 : "memory");
  } else if (DT == kI32 && OP == kSum) {
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.s32 [%0], [%1], %2;" ::"l"(
                     gdst), "r"(smem_addr(smem_src)), "r"(bytes)
                 : "memory");
  } else if (DT == kI32 && OP == kMin) {
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.min.s32 [%0], [%1], %2;" ::"l"(
                     gdst), "r"(smem_addr(smem_src)), "r"(bytes)
                 : "memory");
  } else if (DT == kI32) {
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.max.s32 [%0], [%1], %2;" ::"l"(
                     gdst), "r"(smem_addr(smem_src)), "r"(bytes)
                 : "memory");
  } else if (OP == kMin) {
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.min.bf16 [%0], [%1], %2;" ::"l"(
                     gdst), "r"(smem_addr(smem_src)), "r"(bytes)
                 : "memory");
  } else {
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.max.bf16 [%0], [%1], %2;" ::"l"(
                     gdst), "r"(smem_addr(smem_src)), "r"(bytes)
                 : "memory");
  }
}

// shared -> global bulk copy, tracked by bulk async-groups
__device__ __forceinline__ void bulk_store(void* gdst, const void* smem_src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(smem_addr(smem_src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bulk_wait_read_dyn(int n) {
  switch (n) {
    case 0: bulk_wait_read<0>(); break;
    case 1: bulk_wait_read<1>(); break;
    case 2: bulk_wait_read<2>(); break;
    case 3: bulk_wait_read<3>(); break;
    case 4: bulk_wait_read<4>(); break;
    case 5: bulk_wait_read<5>(); break;
    case 6: bulk_wait_read<6>(); break;
    default: bulk_wait_read<7>(); break;
  }
}

__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// order this thread's generic-proxy shared-memory writes before later
// async-proxy (bulk copy) reads of them
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Named barrier that also ORs a predicate over the participating threads:
// every thread gets the same answer.
__device__ __forceinline__ bool named_bar_or(int id, int nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, %2, %3, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t sm_id() {
  uint32_t s;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(s));
  return s;
}

__device__ __forceinline__ void record_sm(uint32_t* mask) {
  if (mask) {
    uint32_t s = sm_id();
    atomicOr(&mask[(s >> 5) & 7], 1u << (s & 31));
  }
}

// 128-bit global accesses with the streaming (evict-first) cache policy:
// every byte of this path is read or written exactly once.
__device__ __forceinline__ uint4 ld_global_v4(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ void st_global_v4(void* p, uint4 v) {
  __stcs(reinterpret_cast<uint4*>(p), v);
}

// Bounded wait on an mbarrier phase. Gives up when another thread of the CTA
// has flagged an abort, or after `timeout_ns` of %globaltimer time, in which
// case it flags the abort and records a timeout in the status word.
static __device__ __noinline__ bool wait_bounded_slow(uint64_t* bar, uint32_t parity,
                                               volatile int* abort_flag, uint64_t timeout_ns,
                                               int* status, bool honour_abort) {
  uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (honour_abort && *abort_flag) return false;
    if ((i & 31) == 0 && global_ns() - t0 > timeout_ns) {
      *abort_flag = 1;
      atomicCAS(status, 0, kStatusTimeout);
      return false;
    }
  }
}

// The common case (the phase has already completed) costs one try_wait and
// no call; only a wait that has to spin takes the bounded slow path.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity,
                                             volatile int* abort_flag, uint64_t timeout_ns,
                                             int* status, bool honour_abort) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_bounded_slow(bar, parity, abort_flag, timeout_ns, status, honour_abort);
}

// ------------------------------------------------------------------ folds
// R = left fold in ascending rank order. fp32 adds round to nearest (no
// contraction: there is no multiply); min/max keep the earlier rank on ties;
// bf16 widens exactly to fp32 and is rounded once, to nearest even, at the end;
// int32 sums wrap.
template <int OP>
__device__ __forceinline__ float step_f32(float acc, float x) {
  if (OP == kSum) return __fadd_rn(acc, x);
  if (OP == kMin) return (x < acc) ? x : acc;
  return (x > acc) ? x : acc;
}

template <int OP>
__device__ __forceinline__ int32_t step_i32(int32_t acc, int32_t x) {
  if (OP == kSum) return static_cast<int32_t>(static_cast<uint32_t>(acc) + static_cast<uint32_t>(x));
  if (OP == kMin) return (x < acc) ? x : acc;
  return (x > acc) ? x : acc;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

template <int DT, int OP>
struct Fold;

template <int OP>
struct Fold<kF32, OP> {
  float a[4];
  __device__ __forceinline__ void init(uint4 u) {
    a[0] = __uint_as_float(u.x);
    a[1] = __uint_as_float(u.y);
    a[2] = __uint_as_float(u.z);
    a[3] = __uint_as_float(u.w);
  }
  __device__ __forceinline__ void add(uint4 u) {
    a[0] = step_f32<OP>(a[0], __uint_as_float(u.x));
    a[1] = step_f32<OP>(a[1], __uint_as_float(u.y));
    a[2] = step_f32<OP>(a[2], __uint_as_float(u.z));
    a[3] = step_f32<OP>(a[3], __uint_as_float(u.w));
  }
  __device__ __forceinline__ uint4 out() const {
    return make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                      __float_as_uint(a[3]));
  }
};

template <int OP>
struct Fold<kBF16, OP> {
  float a[8];
  __device__ __forceinline__ void init(uint4 u) {
    a[0] = bf16_lo(u.x); a[1] = bf16_hi(u.x);
    a[2] = bf16_lo(u.y); a[3] = bf16_hi(u.y);
    a[4] = bf16_lo(u.z); a[5] = bf16_hi(u.z);
    a[6] = bf16_lo(u.w); a[7] = bf16_hi(u.w);
  }
  __device__ __forceinline__ void add(uint4 u) {
    a[0] = step_f32<OP>(a[0], bf16_lo(u.x)); a[1] = step_f32<OP>(a[1], bf16_hi(u.x));
    a[2] = step_f32<OP>(a[2], bf16_lo(u.y)); a[3] = step_f32<OP>(a[3], bf16_hi(u.y));
    a[4] = step_f32<OP>(a[4], bf16_lo(u.z)); a[5] = step_f32<OP>(a[5], bf16_hi(u.z));
    a[6] = step_f32<OP>(a[6], bf16_lo(u.w)); a[7] = step_f32<OP>(a[7], bf16_hi(u.w));
  }
  __device__ __forceinline__ uint4 out() const {
    return make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]),
                      pack_bf16x2(a[6], a[7]));
  }
};

template <int OP>
struct Fold<kI32, OP> {
  int32_t a[4];
  __device__ __forceinline__ void init(uint4 u) {
    a[0] = static_cast<int32_t>(u.x);
    a[1] = static_cast<int32_t>(u.y);
    a[2] = static_cast<int32_t>(u.z);
    a[3] = static_cast<int32_t>(u.w);
  }
  __device__ __forceinline__ void add(uint4 u) {
    a[0] = step_i32<OP>(a[0], static_cast<int32_t>(u.x));
    a[1] = step_i32<OP>(a[1], static_cast<int32_t>(u.y));
    a[2] = step_i32<OP>(a[2], static_cast<int32_t>(u.z));
    a[3] = step_i32<OP>(a[3], static_cast<int32_t>(u.w));
  }
  __device__ __forceinline__ uint4 out() const {
    return make_uint4(static_cast<uint32_t>(a[0]), static_cast<uint32_t>(a[1]),
                      static_cast<uint32_t>(a[2]), static_cast<uint32_t>(a[3]));
  }
};

// Sums on the packed fp32 pipe: add.rn.f32x2 rounds each half to nearest
// exactly as two scalar adds do, so the fold (ascending rank, fp32, one final
// rounding for bf16) is unchanged; each instruction adds two lanes.
__device__ __forceinline__ uint64_t f32x2_pair(uint32_t lo, uint32_t hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}
__device__ __forceinline__ void f32x2_split(uint64_t v, uint32_t& lo, uint32_t& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=r"(lo), "=r"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t f32x2_add_rn(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

struct PackedSumF32 {
  uint64_t a[2];
  __device__ __forceinline__ void init(uint4 u) {
    a[0] = f32x2_pair(u.x, u.y);
    a[1] = f32x2_pair(u.z, u.w);
  }
  __device__ __forceinline__ void add(uint4 u) {
    a[0] = f32x2_add_rn(a[0], f32x2_pair(u.x, u.y));
    a[1] = f32x2_add_rn(a[1], f32x2_pair(u.z, u.w));
  }
  __device__ __forceinline__ uint4 out() const {
    uint4 r;
    f32x2_split(a[0], r.x, r.y);
    f32x2_split(a[1], r.z, r.w);
    return r;
  }
};

struct PackedSumBF16 {
  uint64_t a[4];  // fp32 pairs (element 2j, element 2j+1)
  __device__ __forceinline__ static uint64_t widen(uint32_t w) {
    return f32x2_pair(w << 16, w & 0xFFFF0000u);
  }
  __device__ __forceinline__ void init(uint4 u) {
    a[0] = widen(u.x); a[1] = widen(u.y); a[2] = widen(u.z); a[3] = widen(u.w);
  }
  __device__ __forceinline__ void add(uint4 u) {
    a[0] = f32x2_add_rn(a[0], widen(u.x));
    a[1] = f32x2_add_rn(a[1], widen(u.y));
    a[2] = f32x2_add_rn(a[2], widen(u.z));
    a[3] = f32x2_add_rn(a[3], widen(u.w));
  }
  __device__ __forceinline__ static uint32_t narrow(uint64_t v) {
    uint32_t lo, hi;
    f32x2_split(v, lo, hi);
    return pack_bf16x2(__uint_as_float(lo), __uint_as_float(hi));
  }
  __device__ __forceinline__ uint4 out() const {
    return make_uint4(narrow(a[0]), narrow(a[1]), narrow(a[2]), narrow(a[3]));
  }
};

// bf16 sums with the mixed-precision add of sm_100 and later: add.rn.f32.bf16
// widens one bf16 half of a register (exactly) and adds it to an fp32
// accumulator with one round to nearest, the same bits as widening first and
// then adding; one instruction per element instead of a widening step per
// element plus half a packed add. The first rank is widened exactly (an add
// to zero would turn -0 into +0).
__device__ __forceinline__ float add_bf16_lo(uint32_t w, float c) {
  float d;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tadd.rn.f32.bf16 %0, l, %2;\n\t}"
      : "=f"(d) : "r"(w), "f"(c));
  return d;
}
__device__ __forceinline__ float add_bf16_hi(uint32_t w, float c) {
  float d;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tadd.rn.f32.bf16 %0, h, %2;\n\t}"
      : "=f"(d) : "r"(w), "f"(c));
  return d;
}

struct MixedSumBF16 {
  float a[8];
  __device__ __forceinline__ void init(uint4 u) {
    a[0] = bf16_lo(u.x); a[1] = bf16_hi(u.x);
    a[2] = bf16_lo(u.y); a[3] = bf16_hi(u.y);
    a[4] = bf16_lo(u.z); a[5] = bf16_hi(u.z);
    a[6] = bf16_lo(u.w); a[7] = bf16_hi(u.w);
  }
  __device__ __forceinline__ void add(uint4 u) {
    a[0] = add_bf16_lo(u.x, a[0]); a[1] = add_bf16_hi(u.x, a[1]);
    a[2] = add_bf16_lo(u.y, a[2]); a[3] = add_bf16_hi(u.y, a[3]);
    a[4] = add_bf16_lo(u.z, a[4]); a[5] = add_bf16_hi(u.z, a[5]);
    a[6] = add_bf16_lo(u.w, a[6]); a[7] = add_bf16_hi(u.w, a[7]);
  }
  __device__ __forceinline__ uint4 out() const {
    return make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]), pack_bf16x2(a[4], a[5]),
                      pack_bf16x2(a[6], a[7]));
  }
};

// The fold the streaming kernels use: packed sums where they exist.
template <int DT, int OP>
struct StreamFold {
  using type = Fold<DT, OP>;
};
template <>
struct StreamFold<kF32, kSum> {
  using type = PackedSumF32;
};
template <>
struct StreamFold<kBF16, kSum> {
  using type = PackedSumBF16;
};

// One element of every selected source, folded, stored to every selected
// destination: the element-wise path for window edges and buffers that are
// not 16-byte co-aligned.
template <int COLL, int DT, int OP, int MAXR>
__device__ __forceinline__ void scalar_element(const BasePtrs<MAXR>& p, int nranks,
                                               const Window& w, uint64_t e) {
  constexpr int es = (DT == kBF16) ? 2 : 4;
  const uint64_t so = w.src_off + e * es;
  const uint64_t dso = w.dst_off + e * es;
  const int d0 = w.dst_sel < 0 ? 0 : w.dst_sel;
  const int d1 = w.dst_sel < 0 ? nranks : w.dst_sel + 1;
  if (COLL == kAllGather) {
    const char* s = static_cast<const char*>(p.src[w.src_sel < 0 ? 0 : w.src_sel]) + so;
    if (es == 2) {
      uint16_t v = *reinterpret_cast<const uint16_t*>(s);
      for (int d = d0; d < d1; ++d) *reinterpret_cast<uint16_t*>(static_cast<char*>(p.dst[d]) + dso) = v;
    } else {
      uint32_t v = *reinterpret_cast<const uint32_t*>(s);
      for (int d = d0; d < d1; ++d) *reinterpret_cast<uint32_t*>(static_cast<char*>(p.dst[d]) + dso) = v;
    }
    return;
  }
  if (DT == kF32) {
    float acc = *reinterpret_cast<const float*>(static_cast<const char*>(p.src[0]) + so);
    for (int r = 1; r < nranks; ++r)
      acc = step_f32<OP>(acc, *reinterpret_cast<const float*>(static_cast<const char*>(p.src[r]) + so));
    for (int d = d0; d < d1; ++d) *reinterpret_cast<float*>(static_cast<char*>(p.dst[d]) + dso) = acc;
  } else if (DT == kBF16) {
    float acc = bf16_lo(*reinterpret_cast<const uint16_t*>(static_cast<const char*>(p.src[0]) + so));
    for (int r = 1; r < nranks; ++r)
      acc = step_f32<OP>(acc, bf16_lo(*reinterpret_cast<const uint16_t*>(static_cast<const char*>(p.src[r]) + so)));
    uint16_t h = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
    for (int d = d0; d < d1; ++d) *reinterpret_cast<uint16_t*>(static_cast<char*>(p.dst[d]) + dso) = h;
  } else {
    int32_t acc = *reinterpret_cast<const int32_t*>(static_cast<const char*>(p.src[0]) + so);
    for (int r = 1; r < nranks; ++r)
      acc = step_i32<OP>(acc, *reinterpret_cast<const int32_t*>(static_cast<const char*>(p.src[r]) + so));
    for (int d = d0; d < d1; ++d) *reinterpret_cast<int32_t*>(static_cast<char*>(p.dst[d]) + dso) = acc;
  }
}

// ------------------------------------------------------------------ bulk engine
constexpr int kMaxStages = 32;
constexpr uint64_t kNoChunk = ~0ull;  // end-of-stream marker in a stage's chunk slot

// Head of the dynamic shared memory, ahead of the stages.
struct BulkSmemHead {
  uint64_t full[kMaxStages];      // stage k holds its chunk (tx-count barrier, 1 arrival)
  uint64_t empty[kMaxStages];     // stage k may be refilled
  uint64_t never;                 // test hook: a barrier nothing signals
  uint64_t chunk_of[kMaxStages];  // chunk index carried by stage k, or kNoChunk
  int abort_flag;
};
constexpr int kBarrierRegion = 1024;
static_assert(sizeof(BulkSmemHead) <= kBarrierRegion, "shared-memory head");

// Chunk index -> (window, byte offset, length), for increasing indices.
struct ChunkLocator {
  uint64_t lo, hi;
  int wi;
  Window w;
  __device__ __forceinline__ void init() {
    wi = -1;
    lo = hi = 0;
  }
  __device__ __forceinline__ void locate(const BulkArgs& a, uint64_t c, uint32_t& off,
                                         uint32_t& n) {
    if (c >= hi) {
      do {
        ++wi;
        hi = a.chunk_prefix[wi + 1];
      } while (c >= hi);
      lo = a.chunk_prefix[wi];
      w = a.win[wi];
    }
    off = static_cast<uint32_t>((c - lo) * static_cast<uint64_t>(a.chunk_bytes));
    n = min(static_cast<uint32_t>(a.chunk_bytes), w.bytes - off);
  }
};

// This CTA's chunks in the static orders: a contiguous range (blocked) or
// every gridDim.x-th chunk (cyclic).
struct StaticOrder {
  uint64_t c, end, step;
  __device__ __forceinline__ void init(const BulkArgs& a) {
    if (a.order == kOrderBlocked) {
      c = static_cast<uint64_t>(blockIdx.x) * a.chunks_per_cta;
      end = min(c + a.chunks_per_cta, a.total_chunks);
      step = 1;
    } else {
      c = blockIdx.x;
      end = a.total_chunks;
      step = gridDim.x;
    }
  }
  __device__ __forceinline__ bool next(uint64_t& out) {
    if (c >= end) return false;
    out = c;
    c += step;
    return true;
  }
};

template <int COLL, int DT, int OP>
__device__ __forceinline__ void bulk_scalar_windows(const BulkArgs& a, int ctid, int nct) {
  const uint32_t b = a.nbody + a.cta_first[blockIdx.x];
  const uint32_t e = a.nbody + a.cta_first[blockIdx.x + 1];
  for (uint32_t wi = b; wi < e; ++wi) {
    const Window w = a.win[wi];
    for (uint64_t x = ctid; x < w.bytes / (DT == kBF16 ? 2 : 4); x += nct)
      scalar_element<COLL, DT, OP, kMaxRanks>(a.p, a.nranks, w, x);
  }
}

// Consumers of the per-rank stage layout: a chunk arrives as P consecutive
// stages (rank 0 first); each consumer thread folds its kPerRankVectors
// vectors of every stage into fp32 / int32 registers and, after rank P-1,
// stores the result to every destination. Only 128-bit register stores.
template <int COLL, int DT, int OP>
__device__ __forceinline__ void per_rank_consumers(const BulkArgs& a, BulkSmemHead& h,
                                                   const unsigned char* stage_base, int ctid,
                                                   int nct, int lane) {
  constexpr int V = kPerRankVectors;
  const int S = a.stages;
  const int P = a.nranks;
  const uint32_t chunk = static_cast<uint32_t>(a.chunk_bytes);
  volatile int* abort_flag = &h.abort_flag;
  ChunkLocator loc;
  loc.init();
  uint32_t it = 0, off = 0, n = 0;
  bool ok = true;
  for (;;) {
    typename StreamFold<DT, OP>::type acc[V];
    bool stop = false;
    for (int r = 0; r < P; ++r) {
      const uint32_t k = it % S;
      if (ok) ok = wait_bounded(&h.full[k], (it / S) & 1, abort_flag, a.timeout_ns, a.status, true);
      if (ok && a.inject_timeout_ns && blockIdx.x == 0 && it == 0)
        ok = wait_bounded(&h.never, 0, abort_flag, a.inject_timeout_ns, a.status, true);
      const uint64_t c = (ok && r == 0) ? h.chunk_of[k] : 0;
      if (__any_sync(0xFFFFFFFFu, !ok || c == kNoChunk)) {
        stop = true;
        break;
      }
      if (r == 0) loc.locate(a, c, off, n);
      const uint4* st = reinterpret_cast<const uint4*>(stage_base + static_cast<size_t>(k) * chunk);
      const uint32_t nv = n >> 4;
#pragma unroll
      for (int j = 0; j < V; ++j) {
        const uint32_t v = ctid + j * nct;
        if (v < nv) {
          if (r == 0) acc[j].init(st[v]);
          else acc[j].add(st[v]);
        }
      }
      // the stage's reads (generic proxy) before the producer's next bulk
      // copy into it (async proxy): without the proxy fence the release can
      // overtake reads whose values are still in flight
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&h.empty[k]);
      ++it;
    }
    if (stop) break;
    const uint32_t nv = n >> 4;
    const int d0 = loc.w.dst_sel < 0 ? 0 : loc.w.dst_sel;
    const int d1 = loc.w.dst_sel < 0 ? P : loc.w.dst_sel + 1;
#pragma unroll
    for (int j = 0; j < V; ++j) {
      const uint32_t v = ctid + j * nct;
      if (v < nv) {
        const uint4 res = acc[j].out();
        const uint64_t o = loc.w.dst_off + off + static_cast<uint64_t>(v) * 16;
        for (int d = d0; d < d1; ++d) st_global_v4(static_cast<char*>(a.p.dst[d]) + o, res);
      }
    }
  }
}

template <int COLL, int DT, int OP>
__global__ void __launch_bounds__(32 * (1 + kMaxConsumerWarps), 1)
    bulk_kernel(const __grid_constant__ BulkArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  BulkSmemHead& h = *reinterpret_cast<BulkSmemHead*>(smem);
  volatile int* abort_flag = &h.abort_flag;
  const int S = a.stages;
  const int P = a.nranks;
  const int nsrc = (COLL == kAllGather) ? 1 : P;
  const uint32_t chunk = static_cast<uint32_t>(a.chunk_bytes);
  unsigned char* stage_base = smem + kBarrierRegion;
  unsigned char* result_base = stage_base + static_cast<size_t>(S) * nsrc * chunk;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ncw = a.consumer_warps;
  const bool ag_bulk = (COLL == kAllGather) && a.store_mode == kStoreBulk;

  if (threadIdx.x == 0) {
    for (int k = 0; k < S; ++k) {
      mbar_init(&h.full[k], 1);
      mbar_init(&h.empty[k], ag_bulk ? 1 : ncw);
    }
    mbar_init(&h.never, 1);
    h.abort_flag = 0;
    fence_mbar_init();
  }
  // An early (programmatic dependent) launch gets here while the stream's
  // previous kernel may still run. Before waiting for it, warm L2 with this
  // CTA's first chunks (in the dynamic order they are fixed: blockIdx.x,
  // + gridDim.x, ...). A prefetch writes nothing, and L2 is where every
  // write lands, so a line the previous kernel still writes is never read
  // stale; the chunk table is the host's upload, no kernel's output.
  if (threadIdx.x == 0 && a.order == kOrderDynamic && !(COLL != kAllGather && a.rank_streamed)) {
    ChunkLocator pl;
    pl.init();
    for (int j = 0; j < S; ++j) {
      const uint64_t c = blockIdx.x + static_cast<uint64_t>(j) * gridDim.x;
      if (c >= a.total_chunks) break;
      uint32_t po, pn;
      pl.locate(a, c, po, pn);
      if (COLL == kAllGather) {
        const char* src = static_cast<const char*>(a.p.src[pl.w.src_sel < 0 ? 0 : pl.w.src_sel]);
        bulk_prefetch_l2(src + pl.w.src_off + po, pn);
      } else {
        for (int r = 0; r < P; ++r)
          bulk_prefetch_l2(static_cast<const char*>(a.p.src[r]) + pl.w.src_off + po, pn);
      }
    }
  }
  // Every other global access comes after this wait, which returns once the
  // previous kernel has finished and its writes are visible (at once for an
  // ordinary launch). The next launch may then be scheduled: its CTAs take
  // this SM only after this CTA exits.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) record_sm(a.sm_mask);
  __syncthreads();

  // ---------------- producer: one thread chooses the chunks and issues every
  // bulk load; it tells the consumers which chunk each stage holds
  if (warp == 0) {
    if (lane != 0) return;
    const bool dynamic = a.order == kOrderDynamic;
    ChunkLocator loc;
    loc.init();
    StaticOrder so;
    so.init(a);
    // L2 prefetch ahead of the ring (static orders only: the sequence is known)
    ChunkLocator pf_loc;
    pf_loc.init();
    StaticOrder pf;
    pf.init(a);
    uint32_t pf_pos = 0;
    const bool prefetch = !dynamic && a.prefetch_chunks > 0;
    if (prefetch) {
      uint64_t skip;
      while (pf_pos < static_cast<uint32_t>(S) && pf.next(skip)) ++pf_pos;
    }
    const uint64_t policy = l2_evict_first_policy();
    // dynamic order: a CTA's first chunks fill its ring and are fixed
    // (blockIdx.x, + gridDim.x, ...), so the ring fills without waiting on
    // the counter; the chunks after the first nfixed * gridDim.x are claimed
    const uint32_t nfixed = (COLL != kAllGather && a.rank_streamed) ? max(1, S / P) : S;
    const uint64_t claimed_base = static_cast<uint64_t>(nfixed) * gridDim.x;
    uint32_t taken = 0;
    unsigned long long next_claim =
        dynamic ? claimed_base + atomicAdd(&a.sched[0], 1ull) : 0ull;
    uint32_t it = 0, off, n;
    bool ok = true;
    for (;;) {
      uint64_t c;
      bool more;
      if (dynamic) {
        if (taken < nfixed) {
          c = blockIdx.x + static_cast<uint64_t>(taken) * gridDim.x;
          ++taken;
        } else {
          c = next_claim;
          // claim the following chunk now; its latency hides behind this one
          if (c < a.total_chunks) next_claim = claimed_base + atomicAdd(&a.sched[0], 1ull);
        }
        more = c < a.total_chunks;
      } else {
        more = so.next(c);
      }
      if (prefetch && more) {
        const uint32_t want = it + S + a.prefetch_chunks;
        uint64_t pc;
        while (pf_pos < want && pf.next(pc)) {
          uint32_t po, pn;
          pf_loc.locate(a, pc, po, pn);
          if (COLL == kAllGather) {
            const char* src = static_cast<const char*>(a.p.src[pf_loc.w.src_sel < 0 ? 0 : pf_loc.w.src_sel]);
            bulk_prefetch_l2(src + pf_loc.w.src_off + po, pn);
          } else {
            for (int r = 0; r < nsrc; ++r)
              bulk_prefetch_l2(static_cast<const char*>(a.p.src[r]) + pf_loc.w.src_off + po, pn);
          }
          ++pf_pos;
        }
      }
      const uint32_t k = it % S;
      if (it >= static_cast<uint32_t>(S)) {
        ok = wait_bounded(&h.empty[k], ((it / S) & 1) ^ 1, abort_flag, a.timeout_ns, a.status, true);
        if (!ok) break;
      }
      if (!more) {
        h.chunk_of[k] = kNoChunk;  // published by the arrive's release
        mbar_arrive(&h.full[k]);
        break;
      }
      loc.locate(a, c, off, n);
      if (COLL != kAllGather && a.rank_streamed) {
        // P stages for this chunk, rank 0 first; rank 0's slot carries the index
        h.chunk_of[k] = c;
        bool stream_ok = true;
        for (int r = 0; r < P; ++r) {
          const uint32_t kr = it % S;
          if (r > 0 && it >= static_cast<uint32_t>(S)) {
            stream_ok = wait_bounded(&h.empty[kr], ((it / S) & 1) ^ 1, abort_flag, a.timeout_ns,
                                     a.status, true);
            if (!stream_ok) break;
          }
          mbar_arrive_expect_tx(&h.full[kr], n);
          const char* src = static_cast<const char*>(a.p.src[r]) + loc.w.src_off + off;
          unsigned char* dst = stage_base + static_cast<size_t>(kr) * chunk;
          if (a.load_evict_first) bulk_load_hint(dst, src, n, &h.full[kr], policy);
          else bulk_load(dst, src, n, &h.full[kr]);
          ++it;
        }
        if (!stream_ok) {
          ok = false;
          break;
        }
        continue;
      }
      h.chunk_of[k] = c;
      mbar_arrive_expect_tx(&h.full[k], n * nsrc);
      unsigned char* st = stage_base + static_cast<size_t>(k) * nsrc * chunk;
      if (COLL == kAllGather) {
        const char* src = static_cast<const char*>(a.p.src[loc.w.src_sel < 0 ? 0 : loc.w.src_sel]);
        if (a.load_evict_first) bulk_load_hint(st, src + loc.w.src_off + off, n, &h.full[k], policy);
        else bulk_load(st, src + loc.w.src_off + off, n, &h.full[k]);
      } else {
        for (int r = 0; r < nsrc; ++r) {
          const char* src = static_cast<const char*>(a.p.src[r]) + loc.w.src_off + off;
          unsigned char* dst = st + static_cast<size_t>(r) * chunk;
          if (a.load_evict_first) bulk_load_hint(dst, src, n, &h.full[k], policy);
          else bulk_load(dst, src, n, &h.full[k]);
        }
      }
      ++it;
    }
    if (!ok) {
      // an abort: let every load this thread issued land before the CTA's
      // shared memory goes away (only the last S iterations can be in flight)
      const uint32_t first = it > static_cast<uint32_t>(S) ? it - S : 0;
      for (uint32_t j = first; j < it; ++j)
        wait_bounded(&h.full[j % S], (j / S) & 1, abort_flag, a.timeout_ns, a.status, false);
    }
    if (dynamic) {
      // the last CTA to finish claiming resets the counter for the next launch
      __threadfence();
      if (atomicAdd(&a.sched[1], 1ull) == gridDim.x - 1) {
        atomicExch(&a.sched[0], 0ull);
        atomicExch(&a.sched[1], 0ull);
      }
    }
    return;
  }

  // ---------------- consumers
  const int ctid = threadIdx.x - 32;
  const int nct = ncw * 32;
  ChunkLocator loc;
  loc.init();
  uint32_t it = 0, off, n;
  bool ok = true;

  if (ag_bulk) {
    // all-gather with bulk stores: the stage itself is the shard, read once
    // from memory and stored from shared memory to all P destinations
    if (ctid == 0) {
      for (;;) {
        const uint32_t k = it % S;
        ok = wait_bounded(&h.full[k], (it / S) & 1, abort_flag, a.timeout_ns, a.status, true);
        if (ok && a.inject_timeout_ns && blockIdx.x == 0 && it == 0)
          ok = wait_bounded(&h.never, 0, abort_flag, a.inject_timeout_ns, a.status, true);
        if (!ok) break;
        const uint64_t c = h.chunk_of[k];
        if (c == kNoChunk) break;
        loc.locate(a, c, off, n);
        const unsigned char* st = stage_base + static_cast<size_t>(k) * chunk;
        const int d0 = loc.w.dst_sel < 0 ? 0 : loc.w.dst_sel;
        const int d1 = loc.w.dst_sel < 0 ? P : loc.w.dst_sel + 1;
        fence_proxy_async_smem();
        for (int d = d0; d < d1; ++d)
          bulk_store(static_cast<char*>(a.p.dst[d]) + loc.w.dst_off + off, st, n);
        bulk_commit();
        bulk_wait_read_dyn(a.release_lag);
        if (it >= static_cast<uint32_t>(a.release_lag))
          mbar_arrive(&h.empty[(it - a.release_lag) % S]);
        ++it;
      }
      bulk_wait_read<0>();
    }
    if (!*abort_flag) bulk_scalar_windows<COLL, DT, OP>(a, ctid, nct);
    return;
  }

  if (COLL != kAllGather && a.rank_streamed) {
    per_rank_consumers<COLL, DT, OP>(a, h, stage_base, ctid, nct, lane);
    if (ctid == 0) bulk_wait_read<0>();
    if (!*abort_flag) bulk_scalar_windows<COLL, DT, OP>(a, ctid, nct);
    return;
  }

  const bool bulk_out = (a.store_mode == kStoreBulk);
  for (;;) {
    const uint32_t k = it % S;
    if (ok) ok = wait_bounded(&h.full[k], (it / S) & 1, abort_flag, a.timeout_ns, a.status, true);
    if (ok && a.inject_timeout_ns && blockIdx.x == 0 && it == 0)
      ok = wait_bounded(&h.never, 0, abort_flag, a.inject_timeout_ns, a.status, true);
    const uint64_t c = ok ? h.chunk_of[k] : kNoChunk;
    const unsigned char* st = stage_base + static_cast<size_t>(k) * nsrc * chunk;
    if (!bulk_out) {
      // each warp decides for itself (its lanes agree through the vote)
      if (__any_sync(0xFFFFFFFFu, c == kNoChunk)) break;
      loc.locate(a, c, off, n);
      const uint32_t nv = n >> 4;
      const int d0 = loc.w.dst_sel < 0 ? 0 : loc.w.dst_sel;
      const int d1 = loc.w.dst_sel < 0 ? P : loc.w.dst_sel + 1;
      for (uint32_t v = ctid; v < nv; v += nct) {
        uint4 res;
        if (COLL == kAllGather) {
          res = reinterpret_cast<const uint4*>(st)[v];
        } else {
          typename StreamFold<DT, OP>::type f;
          f.init(reinterpret_cast<const uint4*>(st)[v]);
#pragma unroll 4
          for (int r = 1; r < P; ++r)
            f.add(reinterpret_cast<const uint4*>(st + static_cast<size_t>(r) * chunk)[v]);
          res = f.out();
        }
        const uint64_t o = loc.w.dst_off + off + static_cast<uint64_t>(v) * 16;
        for (int d = d0; d < d1; ++d) st_global_v4(static_cast<char*>(a.p.dst[d]) + o, res);
      }
      fence_proxy_async_smem();  // the stage's reads before its next bulk copy
      __syncwarp();
      if (lane == 0) mbar_arrive(&h.empty[k]);
    } else {
      unsigned char* res_slot = result_base + static_cast<size_t>(it & 1) * chunk;
      if (ctid == 0) bulk_wait_read<1>();  // the slot's previous stores have read it
      // all consumer threads agree whether to stop; this is also the barrier
      // after which the result slot may be overwritten
      if (named_bar_or(1, nct, c == kNoChunk)) break;
      loc.locate(a, c, off, n);
      const uint32_t nv = n >> 4;
      for (uint32_t v = ctid; v < nv; v += nct) {
        typename StreamFold<DT, OP>::type f;
        f.init(reinterpret_cast<const uint4*>(st)[v]);
#pragma unroll 4
        for (int r = 1; r < P; ++r)
          f.add(reinterpret_cast<const uint4*>(st + static_cast<size_t>(r) * chunk)[v]);
        reinterpret_cast<uint4*>(res_slot)[v] = f.out();
      }
      // the stage's reads before its next bulk copy, and the result slot's
      // writes before the bulk stores read it
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&h.empty[k]);
      named_bar_sync(1, nct);
      if (ctid == 0 && !*abort_flag) {
        const int d0 = loc.w.dst_sel < 0 ? 0 : loc.w.dst_sel;
        const int d1 = loc.w.dst_sel < 0 ? P : loc.w.dst_sel + 1;
        for (int d = d0; d < d1; ++d)
          bulk_store(static_cast<char*>(a.p.dst[d]) + loc.w.dst_off + off, res_slot, n);
        bulk_commit();
      }
    }
    ++it;
  }
  // the CTA may leave once its bulk stores have read shared memory: their
  // writes are complete and visible when the grid is (to the next kernel on
  // the stream, an event, the host); waiting for each write here only delays
  // the grid's last CTA
  if (ctid == 0) bulk_wait_read<0>();
  if (!*abort_flag) bulk_scalar_windows<COLL, DT, OP>(a, ctid, nct);
}

// ------------------------------------------------------------------ TMA-reduce engine
// The reduction itself offloaded to the copy hardware, as the shard-in of the
// T-CCL description does: for each chunk, rank 0's data is bulk-stored into
// the owner's buffer, then ranks 1 .. P-1 are bulk-reduced into it in
// ascending order. For allreduce the final chunk is then loaded once and
// bulk-stored to every other rank. No thread touches the data. Types the
// hardware reduces exactly in this order: fp32 add (round to nearest), int32
// add/min/max, bf16 min/max.
//
// Lane 0 of every warp issues the copies for K chunk slots at once (chunks
// c, c + G, ..., c + (K-1) G of its stream, G = grid x warps), in lock step
// over the ranks: slot 0's operation for rank r, slot 1's, ..., then rank
// r + 1. Each operation is its own bulk async-group, so the group committed
// K groups earlier is the same slot's previous rank: waiting until at most
// K - 1 groups are pending orders the reductions into one owner chunk
// (ascending) while the other K - 1 slots' reductions stay in flight. Each
// slot double-buffers its rank loads; a reduce-scatter gets a third buffer:
// in place, the owner's receive chunk is its own input chunk, which is
// loaded first and kept there, since rank 0's store overwrites it.

__device__ __forceinline__ void bulk_wait_all_dyn(int n) {
  switch (n) {
    case 0: asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); break;
    case 1: asm volatile("cp.async.bulk.wait_group 1;" ::: "memory"); break;
    case 2: asm volatile("cp.async.bulk.wait_group 2;" ::: "memory"); break;
    case 3: asm volatile("cp.async.bulk.wait_group 3;" ::: "memory"); break;
    case 4: asm volatile("cp.async.bulk.wait_group 4;" ::: "memory"); break;
    case 5: asm volatile("cp.async.bulk.wait_group 5;" ::: "memory"); break;
    case 6: asm volatile("cp.async.bulk.wait_group 6;" ::: "memory"); break;
    default: asm volatile("cp.async.bulk.wait_group 7;" ::: "memory"); break;
  }
}

template <int COLL, int DT, int OP>
__global__ void __launch_bounds__(32 * kMaxConsumerWarps, 1)
    reduce_kernel(const __grid_constant__ BulkArgs a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  uint64_t* never = bars + kReduceMaxBarriers;  // test hook: a barrier nothing arrives on
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 8 * (kReduceMaxBarriers + 1));
  unsigned char* buf_base = smem + 1024;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int lanes = blockDim.x >> 5;
  const int K = a.reduce_slots;
  const int NB = a.reduce_bufs;
  const int P = a.nranks;
  const uint32_t chunk = static_cast<uint32_t>(a.chunk_bytes);
  if (threadIdx.x == 0) {
    for (int i = 0; i < lanes * K * NB; ++i) mbar_init(&bars[i], 1);
    mbar_init(never, 1);
    *abort_flag = 0;
    fence_mbar_init();
    record_sm(a.sm_mask);
  }
  __syncthreads();
  if (lane == 0) {
    const int first_bar = warp * K * NB;
    auto bar = [&](int j, int b) { return &bars[first_bar + j * NB + b]; };
    auto buf = [&](int j, int b) {
      return buf_base + static_cast<size_t>(first_bar + j * NB + b) * chunk;
    };
    uint32_t phase = 0;    // bit j * NB + b: parity to wait for on bar(j, b)
    uint32_t pending = 0;  // bit j * NB + b: a load not yet waited for
    auto issue = [&](int j, int b, const char* src, uint32_t n) {
      mbar_arrive_expect_tx(bar(j, b), n);
      bulk_load(buf(j, b), src, n, bar(j, b));
      pending |= 1u << (j * NB + b);
    };
    auto wait_buf = [&](int j, int b) {
      const int bit = j * NB + b;
      const bool done = wait_bounded(bar(j, b), (phase >> bit) & 1, abort_flag, a.timeout_ns,
                                     a.status, true);
      if (done) {
        phase ^= 1u << bit;
        pending &= ~(1u << bit);
      }
      return done;
    };
    // per-slot state of the current K chunks
    uint64_t src_off[kMaxReduceSlots], dst_off[kMaxReduceSlots];
    uint32_t nbytes[kMaxReduceSlots];
    int owner_rank[kMaxReduceSlots], alias[kMaxReduceSlots];
    ChunkLocator loc;
    loc.init();
    bool ok = true, injected = false;
    const uint64_t step = static_cast<uint64_t>(gridDim.x) * lanes;
    for (uint64_t base = static_cast<uint64_t>(blockIdx.x) * lanes + warp;
         base < a.total_chunks && ok; base += step * K) {
      int nvalid = 0;
      for (int j = 0; j < K; ++j) {
        const uint64_t c = base + j * step;
        if (c >= a.total_chunks) break;
        uint32_t off;
        loc.locate(a, c, off, nbytes[j]);
        src_off[j] = loc.w.src_off + off;
        dst_off[j] = loc.w.dst_off + off;
        owner_rank[j] = loc.w.dst_sel < 0 ? 0 : loc.w.dst_sel;
        const char* own = static_cast<const char*>(a.p.dst[owner_rank[j]]) + dst_off[j];
        alias[j] = (NB > 2 && owner_rank[j] > 0 &&
                    own == static_cast<const char*>(a.p.src[owner_rank[j]]) + src_off[j])
                       ? owner_rank[j] : -1;
        ++nvalid;
      }
      bulk_wait_read<0>();  // earlier stores and reductions have read every buffer
      for (int j = 0; j < nvalid; ++j) {
        if (alias[j] > 0)
          issue(j, 2, static_cast<const char*>(a.p.src[alias[j]]) + src_off[j], nbytes[j]);
        issue(j, 0, static_cast<const char*>(a.p.src[0]) + src_off[j], nbytes[j]);
      }
      for (int r = 0; r < P && ok; ++r) {
        for (int j = 0; j < K; ++j) {
          if (j >= nvalid) {
            bulk_commit();  // an empty group keeps every slot K groups apart
            continue;
          }
          // slot j's operation for rank r - 1 is complete (the ascending
          // order; in the arrival order only rank 0's store must land before
          // the reductions, the rest need their buffers read)
          if (r >= 1) {
            if (r == 1 || !a.arrival_order) bulk_wait_all_dyn(K - 1);
            else bulk_wait_read_dyn(K - 1);
          }
          if (r + 1 < P && r + 1 != alias[j])
            issue(j, (r + 1) & 1, static_cast<const char*>(a.p.src[r + 1]) + src_off[j], nbytes[j]);
          if (r == 0 && alias[j] > 0) ok = wait_buf(j, 2);  // the owner's own chunk is safe
          const int b = r == alias[j] ? 2 : (r & 1);
          if (ok && b != 2) ok = wait_buf(j, b);
          if (ok && a.inject_timeout_ns && blockIdx.x == 0 && warp == 0 && !injected) {
            injected = true;
            ok = wait_bounded(never, 0, abort_flag, a.inject_timeout_ns, a.status, true);
          }
          if (!ok) break;
          char* owner = static_cast<char*>(a.p.dst[owner_rank[j]]) + dst_off[j];
          if (r == 0) bulk_store(owner, buf(j, b), nbytes[j]);
          else bulk_reduce<DT, OP>(owner, buf(j, b), nbytes[j]);
          bulk_commit();
        }
      }
      if (!ok) break;
      if (COLL == kAllReduce && P > 1 && !a.anchor_only) {
        // shard-out: each slot's final chunk is loaded once and stored to
        // every other rank; no group is committed in the first loop, so slot
        // j's last reduction has the K - 1 - j later slots' groups after it
        for (int j = 0; j < nvalid; ++j) {
          bulk_wait_all_dyn(K - 1 - j);
          issue(j, 0, static_cast<const char*>(a.p.dst[owner_rank[j]]) + dst_off[j], nbytes[j]);
        }
        for (int j = 0; j < nvalid && ok; ++j) {
          ok = wait_buf(j, 0);
          if (!ok) break;
          for (int d = 0; d < P; ++d)
            if (d != owner_rank[j])
              bulk_store(static_cast<char*>(a.p.dst[d]) + dst_off[j], buf(j, 0), nbytes[j]);
          bulk_commit();
        }
      }
    }
    bulk_wait_all();
    // after an abort, let any load still in flight land before the CTA exits
    for (int bit = 0; bit < K * NB; ++bit)
      if (pending & (1u << bit))
        wait_bounded(&bars[first_bar + bit], (phase >> bit) & 1, abort_flag, a.timeout_ns,
                     a.status, false);
  }
  __syncthreads();
  if (!*abort_flag) bulk_scalar_windows<COLL, DT, OP>(a, threadIdx.x, blockDim.x);
}

// ------------------------------------------------------------------ small engines
template <int MAXW>
__device__ __forceinline__ int find_window(const uint64_t* prefix, int nwin, uint64_t u) {
  int lo = 0, hi = nwin - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= u) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// NP: the rank count fixed at compile time (2 to 8 or 16; 0: a.nranks). The warp engine's
// lane groups then need no run-time division, and both engines' folds (and the
// vec engine's P stores) are unrolled.
template <int COLL, int DT, int OP, int MAXR, int MAXW, bool SHFL, int NP>
__global__ void __launch_bounds__(256) small_kernel(const __grid_constant__ SmallArgs<MAXR, MAXW> a) {
  // an early (programmatic dependent) launch waits here for the stream's
  // previous kernel before any global access (see bulk_kernel)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x == 0) record_sm(a.sm_mask);
  const int P = NP > 0 ? NP : a.nranks;
  const uint64_t nvec = a.vec_prefix[a.nwin];
  const uint64_t nelem = a.elem_prefix[a.nwin];
  const uint64_t gtid = static_cast<uint64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const uint64_t nthr = static_cast<uint64_t>(gridDim.x) * blockDim.x;

  if (SHFL) {
    // one lane per (vector, rank): groups of P lanes, 32 / P groups per warp
    const int lane = threadIdx.x & 31;
    const int vpw = 32 / P;
    const int g = lane / P;
    const int r = lane - g * P;
    const bool lane_used = g < vpw;
    const int base_lane = lane_used ? g * P : 0;
    const uint64_t gwarp = gtid >> 5;
    const uint64_t nwarps = nthr >> 5;
    for (uint64_t base = gwarp * vpw; base < nvec; base += nwarps * vpw) {
      const uint64_t u = base + g;
      const bool valid = lane_used && u < nvec;
      uint4 x = make_uint4(0, 0, 0, 0);
      int wi = 0;
      uint64_t off = 0;
      if (valid) {
        wi = a.nwin == 1 ? 0 : find_window<MAXW>(a.vec_prefix, a.nwin, u);
        off = (u - a.vec_prefix[wi]) * 16;
        const Window& w = a.win[wi];
        if (COLL == kAllGather) {
          if (r == 0)
            x = ld_global_v4(static_cast<const char*>(a.p.src[w.src_sel < 0 ? 0 : w.src_sel]) + w.src_off + off);
        } else {
          x = ld_global_v4(static_cast<const char*>(a.p.src[r]) + w.src_off + off);
        }
      }
      uint4 res;
      if (COLL == kAllGather) {
        res.x = __shfl_sync(0xFFFFFFFFu, x.x, base_lane);
        res.y = __shfl_sync(0xFFFFFFFFu, x.y, base_lane);
        res.z = __shfl_sync(0xFFFFFFFFu, x.z, base_lane);
        res.w = __shfl_sync(0xFFFFFFFFu, x.w, base_lane);
      } else {
        typename StreamFold<DT, OP>::type f;
#pragma unroll (NP > 0 ? NP : 1)
        for (int rr = 0; rr < P; ++rr) {
          uint4 y;
          y.x = __shfl_sync(0xFFFFFFFFu, x.x, base_lane + rr);
          y.y = __shfl_sync(0xFFFFFFFFu, x.y, base_lane + rr);
          y.z = __shfl_sync(0xFFFFFFFFu, x.z, base_lane + rr);
          y.w = __shfl_sync(0xFFFFFFFFu, x.w, base_lane + rr);
          if (rr == 0) f.init(y);
          else f.add(y);
        }
        res = f.out();
      }
      if (valid) {
        const Window& w = a.win[wi];
        if (w.dst_sel < 0) {
          st_global_v4(static_cast<char*>(a.p.dst[r]) + w.dst_off + off, res);
        } else if (r == 0) {
          st_global_v4(static_cast<char*>(a.p.dst[w.dst_sel]) + w.dst_off + off, res);
        }
      }
    }
  } else {
    for (uint64_t u = gtid; u < nvec; u += nthr) {
      const int wi = a.nwin == 1 ? 0 : find_window<MAXW>(a.vec_prefix, a.nwin, u);
      const Window& w = a.win[wi];
      const uint64_t off = (u - a.vec_prefix[wi]) * 16;
      uint4 res;
      if (COLL == kAllGather) {
        res = ld_global_v4(static_cast<const char*>(a.p.src[w.src_sel < 0 ? 0 : w.src_sel]) + w.src_off + off);
      } else {
        typename StreamFold<DT, OP>::type f;
        f.init(ld_global_v4(static_cast<const char*>(a.p.src[0]) + w.src_off + off));
#pragma unroll (NP > 0 ? NP : 8)
        for (int r = 1; r < P; ++r)
          f.add(ld_global_v4(static_cast<const char*>(a.p.src[r]) + w.src_off + off));
        res = f.out();
      }
      const int d0 = w.dst_sel < 0 ? 0 : w.dst_sel;
      const int d1 = w.dst_sel < 0 ? P : w.dst_sel + 1;
      for (int d = d0; d < d1; ++d) st_global_v4(static_cast<char*>(a.p.dst[d]) + w.dst_off + off, res);
    }
  }

  for (uint64_t e = gtid; e < nelem; e += nthr) {
    const int wi = find_window<MAXW>(a.elem_prefix, a.nwin, e);
    scalar_element<COLL, DT, OP, MAXR>(a.p, P, a.win[wi], e - a.elem_prefix[wi]);
  }
}

}  // namespace dev
}  // namespace tccl
