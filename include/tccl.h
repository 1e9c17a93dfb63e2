/*
 * tccl — NCCL-semantics collectives over P logical ranks held in one GPU.
 *
 * Each of the P ranks is a separate buffer in the same GPU's memory. The
 * library plans, lowers and runs allreduce, reduce-scatter and all-gather over
 * those buffers with hand-written sm_103a kernels: a shard-in phase bulk-loads
 * each rank's chunk into a multi-stage shared-memory pipeline and reduces it
 * locally in ascending rank order; a shard-out phase stores the reduced shard,
 * held once on chip, to every destination.
 *
 * Source of the semantics: the T-CCL design as described in the "NCCL M2N vs
 * T-CCL" article (section 2.3 "programming model", 2.4 API table: Group,
 * allreduce / reducescatter / allgather with NCCL semantics, in-place and
 * out-of-place, on a stream), and NCCL's own host API (`ncclAllReduce`), as
 * summarised in the "NCCL Roadmap" post, section "NCCL の API の全体像".
 *
 * Conventions for every call below
 *  - All calls are asynchronous and stream ordered, like NCCL: they enqueue
 *    work on `stream` and return. Buffers must stay valid until that work
 *    completes. A null stream is the legacy default stream.
 *  - The caller owns every buffer. Plain cudaMalloc / framework allocations
 *    are accepted; nothing is registered (the article's section 2.2, "user
 *    buffer compatible").
 *  - The pointer arrays themselves (`sendbufs`, `recvbufs`) are host arrays of
 *    device pointers, read during the call only; the caller may reuse them on
 *    return.
 *  - Every device pointer must be aligned to its element size. Any other
 *    alignment is accepted; 16-byte co-aligned buffers take the fast path.
 *  - The library never aborts, traps or prints (unless the environment
 *    variable TCCL_LOG is set to 1 or 2, which dumps plans to stderr).
 *  - A group is not thread safe: serialise calls on one group. The GPU work of
 *    two calls on one group must not overlap either (as with one NCCL
 *    communicator): calls on different streams need an ordering between them.
 */
#ifndef TCCL_H
#define TCCL_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TCCL_VERSION 1000
#define TCCL_MAX_RANKS 64

typedef struct tcclGroup* tcclGroup_t;

typedef enum {
  tcclSuccess = 0,
  tcclInvalidArgument = 1, /* null/misaligned pointer, bad enum, bad overlap, overflow */
  tcclInvalidUsage = 2,    /* call not valid in the group's state */
  tcclCudaError = 3,       /* a CUDA runtime call or kernel launch failed */
  tcclDeviceTimeout = 4,   /* a device-side wait gave up (reported asynchronously) */
  tcclInternalError = 5
} tcclResult_t;

typedef enum { tcclFloat32 = 0, tcclBfloat16 = 1, tcclInt32 = 2 } tcclDataType_t;

/* Element-wise reductions: the add / min / max the article's section 2.1
 * lists for bulk reductions. Reduction order is ascending rank (see
 * tcclReduceOrder_t for the one exception). */
typedef enum { tcclSum = 0, tcclMin = 1, tcclMax = 2 } tcclRedOp_t;

/* The order in which ranks are combined (tcclConfig_t.reduce_order).
 * Ascending: every engine folds rank 0, then 1, ..., P-1, so results are the
 * same bits on every engine, launch shape and run. Arrival: on the
 * TMA-reduce engine only (the other engines ignore it), ranks 1..P-1 are
 * reduced into the owner chunk with bulk reductions issued back to back, as
 * T-CCL's shard-in describes, and the memory system applies them in the order
 * they arrive. int32 sum/min/max and bf16 min/max are unchanged by order
 * (bit-exact); an fp32 sum may differ from the ascending fold by rounding,
 * within 2 (P-1) 2^-24 sum_r |x_r| of it. */
typedef enum { tcclReduceAscending = 0, tcclReduceArrival = 1 } tcclReduceOrder_t;

/* Which kernel family runs a call (see tcclConfig_t). */
typedef enum {
  tcclEngineAuto = 0,
  tcclEngineBulk = 1, /* TMA cp.async.bulk pipeline: mbarrier stages, reduce, bulk stores */
  tcclEngineWarp = 2, /* small-message path: one lane per (vector, rank), shuffle fold */
  tcclEngineVec = 3,  /* plain 128-bit loads/stores, each lane folds all ranks */
  tcclEngineTmaReduce = 4, /* the copy hardware reduces: rank 0 bulk-stored, ranks 1..P-1
                              bulk-reduced in order, result loaded once and bulk-stored to all;
                              fp32 sum, int32 sum/min/max, bf16 min/max only (other pairs:
                              tcclInvalidUsage); never chosen by Auto */
  tcclEngineCopyOut = 5    /* shard-in on SMs, shard-out on the GPU's copy engines. Allreduce:
                              the message is cut into segments; each segment is reduced by the
                              bulk engine (within the CTA cap) into one anchor rank's receive
                              buffer only, then device-to-device copies on the group's own
                              streams carry it to the other P-1 ranks. All-gather: copies only,
                              no kernel, no SM. Reduce-scatter has no shard-out: one launch of
                              the same register-load fold, shard j into rank j, when every
                              buffer shares its address mod 16 and a shard is a multiple of 16
                              bytes (else the bulk engine). Auto picks it, for calls of at least
                              4 MiB per rank buffer, for allreduce / all-gather when the cap is
                              at most ce_auto_max_cap CTAs, and for reduce-scatter under any cap
                              or uncapped with P <= 4. The segment kernel folds with register
                              loads (128-bit, or 256-bit for P = 2 to 8 or a multiple of 4
                              with every buffer 32-byte aligned past the head) when the send
                              buffers and the anchor's receive buffer share their address mod
                              16, else with the bulk engine's TMA pipeline. */
} tcclEngine_t;

typedef enum {
  tcclStoreAuto = 0,
  tcclStoreBulk = 1, /* reduced chunk staged once in shared memory, P bulk stores */
  tcclStoreVec = 2   /* reduced vector held once in registers, P 128-bit stores */
} tcclStoreMode_t;

/* What one bulk-engine pipeline stage holds. */
typedef enum {
  tcclLayoutAuto = 0,
  tcclLayoutShared = 1,  /* one chunk of every source rank: the fold reads P rows of a stage */
  tcclLayoutPerRank = 2  /* one rank's chunk: P consecutive stages per chunk, partial sums in
                            registers; each bulk copy is a whole stage whatever P is */
} tcclStageLayout_t;

/* How the bulk engine's persistent CTAs share the chunks of a call. */
typedef enum {
  tcclOrderAuto = 0,
  tcclOrderBlocked = 1, /* CTA j takes one contiguous run of chunks */
  tcclOrderCyclic = 2,  /* CTA j takes chunks j, j+G, j+2G, ...: all CTAs sweep the buffers together */
  tcclOrderDynamic = 3  /* CTAs claim chunks from a device counter: faster SMs take more (default) */
} tcclChunkOrder_t;

/*
 * Tuning knobs of a group. Defaults come from tcclGroupCreate (which also
 * reads TCCL_ENGINE, TCCL_SMALL_MAX_BYTES, TCCL_VEC_MAX_BYTES, TCCL_STAGE_BYTES, TCCL_STAGES,
 * TCCL_STORE_MODE, TCCL_CONSUMER_WARPS, TCCL_CTAS_PER_SM,
 * TCCL_WAIT_TIMEOUT_MS, TCCL_CHUNK_ORDER, TCCL_PREFETCH_CHUNKS,
 * TCCL_LOAD_POLICY, TCCL_MAX_CHUNK_BYTES, TCCL_STAGE_LAYOUT, TCCL_CE_STREAMS,
 * TCCL_CE_SEGMENT_BYTES, TCCL_CE_AUTO_MAX_CAP, TCCL_REDUCE_ORDER, TCCL_CE_FOLD,
 * TCCL_CE_TAIL_PERCENT, TCCL_REDUCE_SLOTS, TCCL_CE_AR_STREAMS and TCCL_CE_TAIL_STREAMS once). Zero in a field
 * means "library default".
 *
 * Bulk-engine shape: stage_bytes, stages and max_chunk_bytes default to 64 KiB,
 * 8 and 16 KiB, and a call uses them as given (stages reduced to what shared
 * memory holds), with one exception: while all three hold exactly those
 * defaults, an uncapped, out-of-place allreduce on the bulk engine's shared
 * stage layout that moves 2 * P * S >= 512 MiB keeps about 96 KiB of loads in
 * flight per CTA instead: chunks of 48 KiB / P bytes (at least 6 KiB, at most
 * max_chunk_bytes) and 96 KiB / (P * chunk) stages (at least 2), which
 * streamed 0.5-1% faster on GB300 than a full ring.
 */
typedef struct {
  int engine;              /* tcclEngine_t */
  size_t small_max_bytes;  /* Auto picks the warp engine at or below this many bytes per rank buffer
                              (0: 64 KiB for P >= 5, 128 KiB for fewer ranks) */
  size_t vec_max_bytes;    /* ... and the vec engine up to this many (uncapped calls only) */
  int stage_bytes;         /* bulk engine: shared-memory bytes of one pipeline stage (all sources of one chunk) */
  int stages;              /* bulk engine: pipeline depth (reduced to what shared memory holds) */
  int store_mode;          /* tcclStoreMode_t */
  int consumer_warps;      /* bulk engine: reducing warps per CTA, 1..16 (one more warp issues loads) */
  int ctas_per_sm;         /* bulk engine: resident CTAs per SM the grid is sized for (1 or 2) */
  double wait_timeout_ms;  /* device-side bound on every wait before it reports tcclDeviceTimeout */
  int chunk_order;         /* bulk engine: tcclChunkOrder_t */
  int prefetch_chunks;     /* bulk engine: chunks prefetched into L2 beyond the shared-memory ring
                              (-1 in SetConfig keeps the library default, 0 turns it off) */
  int load_policy;         /* bulk engine: L2 policy of bulk loads: 0 default, 1 evict-first, 2 evict-normal */
  size_t max_chunk_bytes;  /* bulk engine: upper bound on bytes per source per chunk */
  int stage_layout;        /* bulk engine: tcclStageLayout_t */
  int ce_streams;          /* copy-out engine: internal copy streams, 1..8 (default 4) */
  size_t ce_segment_bytes; /* copy-out engine: most bytes per rank in one segment (default
                              28 MiB; a call is cut into at least four segments of at least
                              4 MiB where it can be; rounded down to a multiple of 256) */
  int ce_auto_max_cap;     /* Auto picks the copy-out engine for caps up to this many CTAs
                              (0: by the rank count, 4/7 of the SMs for P <= 2, 5/12 for P = 3
                              and 4, 7/16 for P >= 5; negative: never) */
  int reduce_order;        /* tcclReduceOrder_t (default ascending) */
  int ce_fold;             /* copy-out allreduce, the kernel that folds each segment into the anchor:
                              0 or 1: the register-load fold where every send buffer
                              shares its address mod 16 with the anchor's receive buffer, else the
                              bulk engine's TMA pipeline; 2: always the TMA pipeline (with the
                              group's stage layout and shape); 3: the TMA-reduce engine, rank 0
                              bulk-stored and ranks 1..P-1 bulk-reduced into the anchor in order
                              (no thread touches the data; with the copy engines' shard-out, no
                              thread touches it anywhere), for the pairs that engine supports
                              (fp32 sum, int32 sum/min/max, bf16 min/max), else as 0 */
  int ce_tail_percent;     /* copy-out allreduce: the last segment's length as a percentage of
                              the others (1..100; 0: default 100, equal segments). The number
                              of segments stays the same and the others grow to cover the rest
                              (past ce_segment_bytes if need be): the last segment's copies
                              overlap no fold, so a shorter last segment shortens the tail */
  int reduce_slots;        /* TMA-reduce engine: chunks each issuing thread keeps in flight,
                              1..8 (0: default 4); its chunk size is max_chunk_bytes when that
                              is set, else 8 KiB */
  int ce_ar_streams;       /* copy-out allreduce: copy streams that carry each segment but the
                              last (those copies run beside the next segment's fold, which they
                              slow down); 0: one per 112 / (P - 1) CTAs of the cap (one per 16
                              for P = 8), rounded, at least one (ce_streams uncapped); at most
                              ce_streams */
  int ce_tail_streams;     /* copy-out allreduce: copy streams that carry the last segment (its
                              copies run beside nothing); 0: ce_streams; at most ce_streams */
} tcclConfig_t;

/* What the last launch on a group looked like. */
typedef struct {
  int engine;          /* tcclEngine_t actually used (never Auto); 0 if nothing was launched */
  int store_mode;      /* tcclStoreMode_t actually used */
  int ctas;            /* grid size */
  int threads;         /* threads per CTA */
  int stages;          /* bulk engine pipeline depth (0 otherwise) */
  int chunk_bytes;     /* bulk engine bytes per source per chunk (0 otherwise) */
  int windows;         /* physical windows in the lowered plan */
  int tasks;           /* logical tasks in the plan */
  size_t smem_bytes;   /* dynamic shared memory per CTA */
  int chunk_order;     /* bulk engine: tcclChunkOrder_t used (0 otherwise) */
  uint64_t total_chunks; /* bulk engine: chunks per source in the call */
  int stage_layout;    /* bulk engine: tcclStageLayout_t used (0 otherwise) */
  int ce_segments;     /* copy-out engine: kernel launches (segments) of the call (0 otherwise) */
  int ce_copies;       /* copy-out engine: device-to-device copies enqueued (0 otherwise) */
  int ce_wide_folds;   /* copy-out engine: register-fold launches that read with 256-bit loads
                          (P = 2 to 8 or a multiple of 4, every buffer 32-byte aligned past the head; the same
                          bits as the 128-bit loads, which TCCL_ANCHOR_WIDE=0 in the process's
                          environment keeps); 0 otherwise */
} tcclLaunchInfo_t;

const char* tcclGetErrorString(tcclResult_t r);
tcclResult_t tcclGetVersion(int* version);

/*
 * Create a group of `nranks` logical ranks (1 .. TCCL_MAX_RANKS) on the
 * current CUDA device (the article's `tcl::Group::create`, single-process
 * mode). Allocates a few hundred bytes of device memory for the group's
 * status word and plan tables. Returns tcclInvalidArgument for a bad
 * `nranks` or null `out`, tcclCudaError if the device cannot be queried.
 */
tcclResult_t tcclGroupCreate(int nranks, tcclGroup_t* out);

/* Frees the group and its device memory. Synchronises the device first. */
tcclResult_t tcclGroupDestroy(tcclGroup_t g);

tcclResult_t tcclGroupGetConfig(tcclGroup_t g, tcclConfig_t* cfg);
/* Replaces the group's tuning; cached plans are dropped. */
tcclResult_t tcclGroupSetConfig(tcclGroup_t g, const tcclConfig_t* cfg);

/*
 * Allreduce (the article's `tcl::allreduce(sendbuf, recvbuf, count, op,
 * stream)`, one buffer per logical rank):
 *   recvbufs[r][i] = op-fold over k = 0..P-1 (ascending) of sendbufs[k][i],
 *   for every rank r and every i < count.
 * `count` is elements per rank. fp32 and bf16 accumulate in fp32; bf16 is
 * rounded once at the end, to nearest even. int32 sums wrap.
 * In-place: recvbufs[r] == sendbufs[r] (per rank; mixing is allowed).
 * Any other overlap between a recv buffer and another buffer is
 * tcclInvalidArgument; send buffers may overlap each other.
 * `cta_cap` > 0 bounds the number of CTAs (and so SMs) the call occupies;
 * <= 0 means uncapped. count == 0 returns tcclSuccess without a launch.
 * With the copy-out engine (tcclEngineCopyOut; Auto picks it for large capped
 * calls) the call also uses the group's internal copy streams. They join
 * `stream` through events before the call returns, so work queued on
 * `stream` afterwards sees every rank's result; the call stays capturable
 * into a CUDA graph on `stream`. Calls on different user streams that share
 * a group share those copy streams too (their order between such calls is
 * the order of the calls).
 * The first call of a new shape (count, datatype, cap, the buffers' address
 * mod 16) plans it and, for the bulk engine, uploads its tables with a
 * synchronous copy; the first copy-out call creates the group's copy streams
 * and events. Make those first calls before capturing a CUDA graph; later
 * calls of the same shape allocate nothing and can be captured.
 */
tcclResult_t tcclAllReduce(tcclGroup_t g, const void* const sendbufs[], void* const recvbufs[],
                           size_t count, tcclDataType_t datatype, tcclRedOp_t op,
                           cudaStream_t stream, int cta_cap);

/*
 * Reduce-scatter (the shard-in phase alone):
 *   recvbufs[r][j] = op-fold over k of sendbufs[k][r*recvcount + j].
 * Each send buffer holds P*recvcount elements, each recv buffer recvcount.
 * In-place: recvbufs[r] == sendbufs[r] + r*recvcount elements.
 */
tcclResult_t tcclReduceScatter(tcclGroup_t g, const void* const sendbufs[],
                               void* const recvbufs[], size_t recvcount,
                               tcclDataType_t datatype, tcclRedOp_t op, cudaStream_t stream,
                               int cta_cap);

/*
 * All-gather (the shard-out phase alone: each shard read once, stored to all
 * P destinations):
 *   recvbufs[r][k*sendcount + j] = sendbufs[k][j] for every r.
 * Each send buffer holds sendcount elements, each recv buffer P*sendcount.
 * In-place: sendbufs[r] == recvbufs[r] + r*sendcount elements.
 * The datatype only sets the element size.
 */
tcclResult_t tcclAllGather(tcclGroup_t g, const void* const sendbufs[], void* const recvbufs[],
                           size_t sendcount, tcclDataType_t datatype, cudaStream_t stream,
                           int cta_cap);

/*
 * Waits for all work on the device, then returns (and clears) the group's
 * asynchronous status in *async_status: tcclSuccess, or tcclDeviceTimeout if
 * a kernel gave up on a wait since the last query. Such a kernel skipped the
 * rest of its work, so its outputs are undefined.
 */
tcclResult_t tcclGroupQueryError(tcclGroup_t g, tcclResult_t* async_status);

tcclResult_t tcclGetLastLaunchInfo(tcclGroup_t g, tcclLaunchInfo_t* info);

/*
 * SM-footprint recorder. While enabled, every CTA of every launch sets the
 * bit of the SM it ran on; tcclGroupReadSmRecord synchronises the device,
 * returns the number of distinct SMs seen since the last read and clears the
 * record. Off by default (it adds one atomic per CTA).
 */
tcclResult_t tcclGroupRecordSms(tcclGroup_t g, int enable);
tcclResult_t tcclGroupReadSmRecord(tcclGroup_t g, int* distinct_sms);

/*
 * The same record, launch by launch: each kernel launch made while recording
 * sets bits in a bitmap of its own (up to 64 launches; later ones share the
 * last bitmap). Synchronises the device, writes the distinct SMs of each of
 * the first `max_launches` recorded launches to per_launch[0 ..], the number
 * of launches recorded to *n_launches and the distinct SMs of all of them
 * together to *distinct_sms, then clears the record. A copy-out call (several
 * segment kernels, each within the cap) shows here as several launches.
 * per_launch may be null when max_launches is 0. Errors: tcclInvalidArgument
 * for a null group or output, tcclCudaError if the device cannot be read.
 */
tcclResult_t tcclGroupReadSmRecordLaunches(tcclGroup_t g, int* per_launch, int max_launches,
                                           int* n_launches, int* distinct_sms);

/*
 * Host-only view of the planner and lowering (no GPU needed). Plans and
 * lowers one collective for a device with `sm_count` SMs and
 * `smem_per_block` bytes of opt-in shared memory, as a call with these
 * pointers would be, without launching anything. `coll` is 0 allreduce,
 * 1 reduce-scatter, 2 all-gather; `count` is the per-call count argument.
 * The buffer addresses are only used for their alignment and overlap.
 * Writes up to `max_windows` windows, eight int64 values each:
 *   {cta, src_sel, src_off, dst_sel, dst_off, bytes, scalar, task}:
 * owning CTA (-1 unless the window is element-wise and run by the bulk
 * engine, which binds those to CTAs), source rank or -1 for all ranks, byte
 * offset into the source buffer(s), destination rank or -1, byte offset into
 * the destination buffer(s), window bytes, 1 if the window needs the
 * element-wise (unaligned) path, and the logical task it came from.
 * *n_windows receives the total count, *info the launch shape.
 * Argument errors are reported exactly as the collective call would.
 */
tcclResult_t tcclPlanInspect(int coll, int nranks, const void* const sendbufs[],
                             void* const recvbufs[], size_t count, tcclDataType_t datatype,
                             int cta_cap, int sm_count, int smem_per_block,
                             const tcclConfig_t* cfg, int64_t* windows, int max_windows,
                             int* n_windows, int* n_tasks, tcclLaunchInfo_t* info);

/*
 * Host-only view of the copy-out engine's decisions (no GPU needed), for a
 * call with these arguments on a device with `sm_count` SMs under `cfg`
 * (null: the defaults). The buffer addresses are only used for their
 * alignment and overlap. Outputs:
 *   *copy_out       1 if the call would run on the copy-out engine;
 *   *register_fold  1 if its shard-in would be the register-load fold
 *                   (0: the TMA pipeline for an allreduce; a reduce-scatter
 *                   the fold cannot take runs on the bulk engine, and then
 *                   *copy_out is 0 too);
 *   *segments, *segment_elems  an allreduce's segments and the length of all
 *                   but the last; 1 and `count` for a reduce-scatter on the
 *                   fold; 0 otherwise (an all-gather is copies only);
 *   *wide_folds     how many of those fold launches would read with 256-bit
 *                   loads (the launch info's ce_wide_folds), in this
 *                   process's environment (TCCL_ANCHOR_WIDE).
 * count == 0 and no-op calls report 0 everywhere. Argument errors are
 * reported exactly as the collective call would.
 */
tcclResult_t tcclCopyOutInspect(int coll, int nranks, const void* const sendbufs[],
                                void* const recvbufs[], size_t count, tcclDataType_t datatype,
                                int cta_cap, int sm_count, const tcclConfig_t* cfg, int* copy_out,
                                int* register_fold, int* segments, size_t* segment_elems,
                                int* wide_folds);

/*
 * Test hook for the bounded-wait error path: while enabled, each bulk-engine
 * launch makes its first CTA wait on a barrier that nothing signals, with a
 * `timeout_ms` bound; the CTA then records tcclDeviceTimeout, skips its
 * remaining work and exits normally (no trap, no fault). Other CTAs finish.
 */
tcclResult_t tcclGroupInjectWaitTimeout(tcclGroup_t g, int enable, double timeout_ms);

/*
 * Allreduce fused with RMSNorm (the "NCCL Roadmap" post, section "GENK と
 * Flow", mentions a Device API example that folds a Transformer RMSNorm into
 * one kernel with the reduce-scatter and all-gather). Every rank buffer holds
 * [rows, hidden] activations; afterwards every recv buffer holds
 *   y[t, j] = s[t, j] * rsqrt(mean_k(s[t, k]^2) + eps) * gamma[j],
 * s = the ascending-rank fp32 sum of the sends (never rounded), y rounded once
 * to the datatype (fp32 or bf16). gamma: `hidden` elements of the datatype in
 * device memory. The row's sum of squares is a parallel reduction, so results
 * match a plain evaluation to within one unit in the last place of the output
 * type, not bit for bit.
 * Limits: hidden a multiple of 8 (bf16) or 4 (fp32), at most 16384 (bf16) or
 * 8192 (fp32); every buffer 16-byte aligned; in place allowed as for
 * tcclAllReduce; int32 is tcclInvalidArgument.
 */
tcclResult_t tcclAllReduceRMSNorm(tcclGroup_t g, const void* const sendbufs[],
                                  void* const recvbufs[], size_t rows, size_t hidden,
                                  const void* gamma, float eps, tcclDataType_t datatype,
                                  cudaStream_t stream, int cta_cap);

/*
 * M-to-N reshard between two layouts of one tensor (the M2N collective of the
 * "NCCL M2N vs T-CCL" article, §1.2-§1.4, on logical ranks of one GPU).
 *
 * A layout is a mesh of ranks: `ndims` dimensions `dims` in row-major rank
 * order, holding group ranks [start_rank, start_rank + prod(dims)), and one
 * placement per mesh axis, TCCL_REPLICATE or the tensor dimension that axis
 * shards into equal contiguous blocks. At most one axis may shard (the
 * article's constraint), each sharded dimension must divide evenly, and the
 * source and destination meshes must not share ranks.
 *
 * srcbufs[m] / dstbufs[m] is mesh rank m's local block, contiguous and
 * row-major. Source replicas must hold identical data. Afterwards every
 * destination rank holds exactly the block its layout names. The plan comes
 * from the layouts alone by interval intersection: every piece a destination
 * block needs is read once, from the least-loaded source replica, and written
 * to every destination replica of that block.
 *
 * Engines (the group's tcclConfig_t.engine): with every piece 16-byte
 * co-aligned in every buffer, a bulk ring (one CTA per SM, bulk loads into
 * shared memory, bulk stores to every replica) runs the copies under
 * tcclEngineBulk always, and under Auto when blocks have three or more
 * replicas on average and every row piece is 4 KiB or more; otherwise, and
 * always under tcclEngineWarp or tcclEngineVec, warps copy through
 * registers. A ring wait that runs out is reported by tcclGroupQueryError as
 * tcclDeviceTimeout. As for every call on a group, reshards on different
 * streams need an ordering between them (a plan's ring keeps one work counter).
 *
 * Errors: tcclInvalidArgument for a bad layout, shape, pointer or overlap
 * (destination buffers may not overlap each other or any source), or meshes
 * outside the group's ranks.
 */
#define TCCL_REPLICATE (-1)
#define TCCL_MAX_MESH_DIMS 4
#define TCCL_MAX_TENSOR_DIMS 4
typedef struct {
  int ndims;
  int dims[TCCL_MAX_MESH_DIMS];
  int start_rank;
  int placements[TCCL_MAX_MESH_DIMS];
} tcclLayout_t;

tcclResult_t tcclReshard(tcclGroup_t g, const void* const srcbufs[], const tcclLayout_t* src,
                         void* const dstbufs[], const tcclLayout_t* dst, int tensor_ndims,
                         const size_t* tensor_shape, tcclDataType_t datatype,
                         cudaStream_t stream, int cta_cap);

/*
 * Host-only view of a reshard plan (no GPU needed). Writes up to
 * `max_transfers` transfers, ten int64 values each:
 *   {source mesh rank, destination replica mask, lo[4], hi[4]} (global
 *   coordinates of the piece; unused dimensions 0), and the totals.
 * Buffer addresses are used only for their alignment.
 */
tcclResult_t tcclReshardInspect(const tcclLayout_t* src, const tcclLayout_t* dst,
                                int tensor_ndims, const size_t* tensor_shape,
                                tcclDataType_t datatype, const void* const srcbufs[],
                                void* const dstbufs[], int sm_count, int cta_cap,
                                int64_t* transfers, int max_transfers, int* n_transfers,
                                int64_t* bytes_read, int64_t* bytes_written, int* n_windows);

/*
 * Allreduce for callers that cannot allocate GPU memory (no counterpart in
 * the paper: a convenience of this library).
 *
 * Who needs it: code that must not call cudaMalloc, such as a component
 * running under another framework's memory manager that owns every device
 * allocation, an allocator hook or out-of-memory handler, or a process whose
 * device memory is reserved up front. tcclGroupCreate allocates device memory
 * (a status word and plan tables), so this call takes no group.
 *
 * Computes exactly what tcclAllReduce computes, with the bulk engine, and
 * allocates no device or pinned memory: it calls no cudaMalloc, cudaFree,
 * cudaMallocHost, cudaMallocAsync or other allocating CUDA routine. Its
 * scratch (status word, per-CTA offsets, window table) is one static device
 * array of TCCL_NO_ALLOC_SCRATCH_BYTES that every GPU loading this library
 * holds until the process exits; host-side planning uses ordinary C++ heap
 * memory.
 *  - The first call on a device (with that device current) resolves the
 *    array's device address with cudaGetSymbolAddress and creates one event
 *    and one stream for reading the status word; make that first call before
 *    any stream capture.
 *  - Each call copies its plan from host memory into the array, in stream
 *    order. A call on a stream that is being captured returns
 *    tcclInvalidUsage and enqueues nothing.
 *  - Every call shares the one array and overwrites it with its own plan, so
 *    calls whose work overlaps on the GPU (different streams, or other
 *    threads) race and give undefined results. Serialise them; the function
 *    is not thread safe.
 *  - Plans needing more than TCCL_NO_ALLOC_MAX_CTAS CTAs, or more windows
 *    than the array holds, are rejected with tcclInvalidUsage (TCCL_LOG=1
 *    prints the sizes); every other argument rule is tcclAllReduce's.
 *  - Device-side timeouts: a kernel that gives up on a bounded wait skips
 *    the rest of its work (its outputs are undefined) and records
 *    tcclDeviceTimeout in the array's status word. A later call on the same
 *    device reports it: each call first checks, without waiting, whether the
 *    previous call's kernel has finished and, if so, reads the word. When it
 *    finds a timeout recorded, the call returns tcclDeviceTimeout, launches
 *    nothing and clears the record; call again to run it. A timeout of the
 *    last call is therefore seen by the next call made after that call's
 *    work has finished (for instance after a stream synchronisation).
 *  - Test hook: the environment variable TCCL_NO_ALLOC_INJECT_TIMEOUT_MS > 0
 *    makes the first CTA of each launch wait that many milliseconds on a
 *    barrier nothing signals, so the timeout path can be exercised.
 */
#define TCCL_NO_ALLOC_SCRATCH_BYTES (256 * 1024)
#define TCCL_NO_ALLOC_MAX_CTAS 1024
tcclResult_t tcclAllReduceNoAlloc(int nranks, const void* const sendbufs[],
                                  void* const recvbufs[], size_t count, tcclDataType_t datatype,
                                  tcclRedOp_t op, cudaStream_t stream, int cta_cap);

#ifdef __cplusplus
}
#endif

#endif /* TCCL_H */
