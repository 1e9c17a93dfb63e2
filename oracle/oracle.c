/*
 * CPU oracle for the collectives over P logical rank buffers.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the library calls this code: only the
 * tests, the smoke check and the benchmark's CPU-baseline leg load it. It
 * shares no code, header, table or helper with the CUDA path.
 *
 * What it computes is the plain definition of each collective, with no
 * shards, windows, chunks or reordering:
 *   allreduce:      recv[r][i]        = R(send[0][i], ..., send[P-1][i])     for every r
 *   reduce-scatter: recv[r][j]        = R(send[0][r*rc + j], ..., send[P-1][r*rc + j])
 *   all-gather:     recv[r][k*sc + j] = send[k][j]                           for every r
 * These are the NCCL-semantics collectives the T-CCL host API offers
 * ("NCCL M2N vs T-CCL" article, section 2.4 API table: allreduce,
 * reducescatter, allgather over sendbuf/recvbuf/count/op/stream) with the
 * element-wise add/min/max reductions of the TMA bulk-reduce primitive it
 * builds on (same article, section 2.1). The owner reduces the P
 * contributions locally (section 2.2, reduction localisation).
 *
 * R is a left fold in ascending rank order: acc = x_0, then
 * acc = op(acc, x_r) for r = 1 .. P-1. The pages only say "reduce locally";
 * the fixed ascending order, fp32 accumulation for fp32 and bf16 inputs and a
 * single final round-to-nearest-even to bf16 are this library's stated
 * reading of it.
 *   sum f32 : acc = acc + x      (IEEE binary32, round to nearest; built
 *                                 without fast-math and without contraction)
 *   min     : acc = (x < acc) ? x : acc      (earlier rank wins ties)
 *   max     : acc = (x > acc) ? x : acc
 *   sum i32 : two's-complement wrapping add (done on uint32_t)
 *   bf16    : each input widened to binary32 exactly (bits << 16), folded as
 *             f32, then rounded once to bf16, nearest, ties to even.
 *
 * Loops are element-outer, rank-inner, single threaded. The *_mt variants
 * split the element range over threads and run the same per-element code, so
 * their bits are identical; they exist to time the oracle on all host cores.
 *
 * In-place forms (recv aliasing send the NCCL way) are safe here because
 * every output element is written only after all P inputs it depends on have
 * been read, and no later output reads it.
 */
#include <pthread.h>
#include <stdint.h>
#include <string.h>

enum { OR_F32 = 0, OR_BF16 = 1, OR_I32 = 2 };
enum { OR_SUM = 0, OR_MIN = 1, OR_MAX = 2 };

/* ---- element helpers -------------------------------------------------- */

static float or_bf16_widen(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

/* binary32 -> bf16, round to nearest, ties to even (finite inputs). */
static uint16_t or_bf16_round(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  uint32_t keep_lsb = (u >> 16) & 1u;
  u = u + 0x7FFFu + keep_lsb;
  return (uint16_t)(u >> 16);
}

static float or_fold_f32(int op, float acc, float x) {
  switch (op) {
    case OR_SUM: return acc + x;
    case OR_MIN: return (x < acc) ? x : acc;
    default: return (x > acc) ? x : acc;
  }
}

static int32_t or_fold_i32(int op, int32_t acc, int32_t x) {
  switch (op) {
    case OR_SUM: return (int32_t)((uint32_t)acc + (uint32_t)x);
    case OR_MIN: return (x < acc) ? x : acc;
    default: return (x > acc) ? x : acc;
  }
}

/* reduce element `si` of all P sends, write it to element `di` of `dst` */
static void or_reduce_one(int dtype, int op, int nranks, const void* const* send,
                          uint64_t si, void* dst, uint64_t di) {
  if (dtype == OR_F32) {
    float acc = ((const float*)send[0])[si];
    for (int r = 1; r < nranks; ++r) acc = or_fold_f32(op, acc, ((const float*)send[r])[si]);
    ((float*)dst)[di] = acc;
  } else if (dtype == OR_BF16) {
    float acc = or_bf16_widen(((const uint16_t*)send[0])[si]);
    for (int r = 1; r < nranks; ++r)
      acc = or_fold_f32(op, acc, or_bf16_widen(((const uint16_t*)send[r])[si]));
    ((uint16_t*)dst)[di] = or_bf16_round(acc);
  } else {
    int32_t acc = ((const int32_t*)send[0])[si];
    for (int r = 1; r < nranks; ++r) acc = or_fold_i32(op, acc, ((const int32_t*)send[r])[si]);
    ((int32_t*)dst)[di] = acc;
  }
}

static int or_elem_size(int dtype) { return dtype == OR_BF16 ? 2 : 4; }

static int or_check(int dtype, int op, int nranks, const void* const* send, void* const* recv) {
  if (dtype < OR_F32 || dtype > OR_I32) return -1;
  if (op < OR_SUM || op > OR_MAX) return -1;
  if (nranks < 1 || nranks > 1024 || !send || !recv) return -1;
  for (int r = 0; r < nranks; ++r)
    if (!send[r] || !recv[r]) return -1;
  return 0;
}

/* ---- allreduce ------------------------------------------------------- */

static void or_allreduce_range(int dtype, int op, int nranks, const void* const* send,
                               void* const* recv, uint64_t begin, uint64_t end) {
  int es = or_elem_size(dtype);
  for (uint64_t i = begin; i < end; ++i) {
    /* reduce into rank 0's output, then copy that one value to the others */
    union { float f; uint16_t h; int32_t i; } v;
    or_reduce_one(dtype, op, nranks, send, i, &v, 0);
    for (int r = 0; r < nranks; ++r) memcpy((char*)recv[r] + i * (uint64_t)es, &v, (size_t)es);
  }
}

int oracle_allreduce(int dtype, int op, int nranks, uint64_t count, const void* const* send,
                     void* const* recv) {
  if (or_check(dtype, op, nranks, send, recv)) return -1;
  or_allreduce_range(dtype, op, nranks, send, recv, 0, count);
  return 0;
}

/* ---- reduce-scatter -------------------------------------------------- */

static void or_reduce_scatter_range(int dtype, int op, int nranks, uint64_t recvcount,
                                    const void* const* send, void* const* recv,
                                    uint64_t jbegin, uint64_t jend) {
  for (int s = 0; s < nranks; ++s)
    for (uint64_t j = jbegin; j < jend; ++j)
      or_reduce_one(dtype, op, nranks, send, (uint64_t)s * recvcount + j, recv[s], j);
}

int oracle_reduce_scatter(int dtype, int op, int nranks, uint64_t recvcount,
                          const void* const* send, void* const* recv) {
  if (or_check(dtype, op, nranks, send, recv)) return -1;
  or_reduce_scatter_range(dtype, op, nranks, recvcount, send, recv, 0, recvcount);
  return 0;
}

/* ---- all-gather ------------------------------------------------------ */

static void or_allgather_range(int elem_size, int nranks, uint64_t sendcount,
                               const void* const* send, void* const* recv, uint64_t jbegin,
                               uint64_t jend) {
  for (int k = 0; k < nranks; ++k)
    for (uint64_t j = jbegin; j < jend; ++j)
      for (int r = 0; r < nranks; ++r)
        memmove((char*)recv[r] + ((uint64_t)k * sendcount + j) * (uint64_t)elem_size,
                (const char*)send[k] + j * (uint64_t)elem_size, (size_t)elem_size);
}

int oracle_allgather(int elem_size, int nranks, uint64_t sendcount, const void* const* send,
                     void* const* recv) {
  if (elem_size != 2 && elem_size != 4) return -1;
  if (or_check(OR_F32, OR_SUM, nranks, send, recv)) return -1;
  or_allgather_range(elem_size, nranks, sendcount, send, recv, 0, sendcount);
  return 0;
}

/* ---- threaded variants (same per-element code, split element ranges) -- */

typedef struct {
  int which; /* 0 AR, 1 RS, 2 AG */
  int dtype, op, nranks, elem_size;
  uint64_t n; /* count / recvcount / sendcount */
  const void* const* send;
  void* const* recv;
  uint64_t begin, end;
} or_job;

static void or_run(const or_job* j) {
  if (j->which == 0)
    or_allreduce_range(j->dtype, j->op, j->nranks, j->send, j->recv, j->begin, j->end);
  else if (j->which == 1)
    or_reduce_scatter_range(j->dtype, j->op, j->nranks, j->n, j->send, j->recv, j->begin,
                            j->end);
  else
    or_allgather_range(j->elem_size, j->nranks, j->n, j->send, j->recv, j->begin, j->end);
}

static void* or_thread(void* a) {
  or_run((const or_job*)a);
  return 0;
}

static int or_parallel(or_job proto, int nthreads) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if ((uint64_t)nthreads > proto.n / 4096 + 1) nthreads = (int)(proto.n / 4096 + 1);
  or_job jobs[256];
  pthread_t th[256];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = proto;
    jobs[t].begin = proto.n * (uint64_t)t / (uint64_t)nthreads;
    jobs[t].end = proto.n * (uint64_t)(t + 1) / (uint64_t)nthreads;
  }
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&th[t], 0, or_thread, &jobs[t]) != 0) break;
    started = t;
  }
  or_run(&jobs[0]);
  for (int t = 1; t <= started; ++t) pthread_join(th[t], 0);
  for (int t = started + 1; t < nthreads; ++t) or_run(&jobs[t]);
  return nthreads;
}

/* Each returns the number of threads used, or -1 on bad arguments. */
int oracle_allreduce_mt(int dtype, int op, int nranks, uint64_t count, const void* const* send,
                        void* const* recv, int nthreads) {
  if (or_check(dtype, op, nranks, send, recv)) return -1;
  or_job j = {0, dtype, op, nranks, or_elem_size(dtype), count, send, recv, 0, 0};
  return or_parallel(j, nthreads);
}

int oracle_reduce_scatter_mt(int dtype, int op, int nranks, uint64_t recvcount,
                             const void* const* send, void* const* recv, int nthreads) {
  if (or_check(dtype, op, nranks, send, recv)) return -1;
  or_job j = {1, dtype, op, nranks, or_elem_size(dtype), recvcount, send, recv, 0, 0};
  return or_parallel(j, nthreads);
}

int oracle_allgather_mt(int elem_size, int nranks, uint64_t sendcount, const void* const* send,
                        void* const* recv, int nthreads) {
  if (elem_size != 2 && elem_size != 4) return -1;
  if (or_check(OR_F32, OR_SUM, nranks, send, recv)) return -1;
  or_job j = {2, OR_F32, OR_SUM, nranks, elem_size, sendcount, send, recv, 0, 0};
  return or_parallel(j, nthreads);
}
