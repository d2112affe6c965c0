/*
 * sparse_attn.h -- C ABI of libsparse_attn: per-head-budget block-sparse
 * attention on one GB300 (sm_103a).
 *
 * The library computes one attention layer with block-granularity top-k
 * sparsity where every query head has its own block budget:
 *
 *   plan     per-head budgets by Max-Min budget shifting around a uniform
 *            budget, and a greedy longest-first (LPT) schedule of
 *            (head, query-block) work items over persistent workers.
 *            Source: "S-HPLB: Efficient LLM Attention Serving via
 *            Sparsity-Aware Head Parallelism Load Balance" -- Italian summary,
 *            "Metodologia" A ("Strategia Max-Min (Budget Shifting)") and B
 *            ("Algoritmo Greedy"); Chinese summary 2.1 and 2.2.
 *   score    (Index) mean-pooled query-block x key-block scores.
 *   select   (Select) per-row top-k_h blocks, always keeping the sink block 0
 *            and the diagonal block.
 *   forward  (Attention) online-softmax attention over only the selected
 *            blocks, with grouped-query KV sharing.
 *            The Index / Select / Attention split is the one of "Unifying
 *            Sparse Attention with Hierarchical Memory for Scalable
 *            Long-Context LLM Serving" (Spin), "Abstracción de Partición
 *            Unificada"; block granularity, the sink block and the
 *            streaming / retrieval head split are from "Riepilogo Tecnico:
 *            Fluxion", "Intuizioni Chiave" 1 and 2.
 *
 * Conventions
 *  - Every call returns sa_status; none aborts, throws or prints.
 *  - Device pointers are caller-owned (allocated by the caller, e.g. by
 *    PyTorch).  The library owns only the opaque sa_plan, including the
 *    device copy of its schedule made by sparse_attn_plan_upload.
 *  - Device calls are asynchronous on the given stream (NULL = the legacy
 *    default stream).  Argument errors are reported before anything is
 *    launched; errors the device detects (corrupt block indices, timeouts
 *    of bounded waits) are OR-ed into a caller-supplied int32 status word
 *    (SA_DEV_* bits) which the caller reads after synchronising.
 *  - Layouts (row-major, contiguous, bfloat16 unless stated):
 *      prefill  Q [Hq][S][d], K and V [Hkv][S][d], O [Hq][S][d];
 *      decode   q [Bt][Hq][d], K and V [Bt][Hkv][L][d], o [Bt][Hq][d].
 *    Query head h reads KV head h / (Hq/Hkv).  A block is B consecutive
 *    tokens; nb = S / B (or L / B).
 *  - Supported: bf16, d in {64, 128}; prefill B in {64, 128} with
 *    B*d*2 bytes per block as a TMA box; decode B = 32; S % B == 0.
 *    Other shapes return SA_ERR_UNSUPPORTED.
 */
#ifndef SPARSE_ATTN_H
#define SPARSE_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (the same type as cudaStream_t). */
typedef struct CUstream_st* sa_stream_t;

typedef enum sa_status {
  SA_OK = 0,
  SA_ERR_INVALID_ARG = 1,    /* null pointer, bad enum, out-of-range scalar */
  SA_ERR_SHAPE = 2,          /* inconsistent sizes (S % B, Hq % Hkv, kmax) */
  SA_ERR_UNSUPPORTED = 3,    /* valid but not implemented (d, B, mode)     */
  SA_ERR_CUDA = 4,           /* a CUDA runtime / driver call failed        */
  SA_ERR_DEVICE_CHECK = 5,   /* reserved: device status word reported bits */
  SA_ERR_DEVICE_TIMEOUT = 6, /* reserved: a bounded device wait gave up    */
  SA_ERR_NO_MEMORY = 7,      /* host or device allocation failed           */
  SA_ERR_NOT_UPLOADED = 8    /* plan used on the device before upload      */
} sa_status;

enum { SA_MODE_PREFILL = 0, SA_MODE_DECODE = 1 };

/* Work schedules of (head, query-block) items over persistent workers. */
enum {
  SA_SCHED_LPT = 0,          /* cost-descending greedy, least-loaded worker  */
  SA_SCHED_LPT_GROUPED = 1,  /* the same greedy, walked KV group by KV group */
  SA_SCHED_HEAD_ORDER = 2    /* naive: items in head order, equal chunks     */
};

enum { SA_HEAD_RETRIEVAL = 0, SA_HEAD_STREAMING = 1 };

/* Element type of the attention output. */
enum { SA_DTYPE_BF16 = 0, SA_DTYPE_F32 = 1 };

/* Bits of the device status word. */
enum {
  SA_DEV_BAD_INDEX = 1,      /* a block index outside [0, i] was clamped     */
  SA_DEV_BAD_COUNT = 2,      /* a block count outside [1, min(kmax,i+1)]     */
  SA_DEV_TIMEOUT = 4,        /* a bounded wait gave up; outputs are invalid  */
  SA_DEV_BAD_ITEM = 8,       /* a schedule entry outside the item range      */
  SA_DEV_BAD_LAUNCH = 16,    /* the kernel found its shared memory misaligned
                                and did nothing; outputs are not written     */
  SA_DEV_RANGE = 32          /* rows beyond the tensor-core pass's range
                                (a row sum above 2^126 or O overflowed) could
                                not all be recomputed exactly: a worker list
                                longer than 32768 items; outputs invalid     */
};

typedef struct sa_shape {
  int64_t seq_len;       /* S (prefill) or cache length L (decode)          */
  int32_t block;         /* B, tokens per block                             */
  int32_t num_q_heads;   /* Hq                                              */
  int32_t num_kv_heads;  /* Hkv (divides Hq)                                */
  int32_t head_dim;      /* d                                               */
  int32_t batch;         /* decode: sequences Bt; prefill: must be 1        */
  int32_t mode;          /* SA_MODE_PREFILL or SA_MODE_DECODE               */
} sa_shape;

typedef struct sa_plan_params {
  const int32_t* demand;    /* [Hq] per-head block demand d_h from offline
                               calibration, or NULL: all budgets = k_uniform.
                               Prefill only (must be NULL for decode).      */
  int32_t k_uniform;        /* uniform starting budget, blocks per row;
                               k_min <= k_uniform <= max(nb, k_min)          */
  int32_t k_min;            /* smallest budget a head may be shifted to; >= 2
                               (the sink and diagonal blocks)               */
  const uint8_t* head_kind; /* decode: [Hq] SA_HEAD_*; NULL = all retrieval.
                               Must be NULL for prefill.                    */
  int32_t window_blocks;    /* decode: recent blocks a streaming head keeps
                               besides block 0 (>= 1 when any streaming)    */
  int32_t num_workers;      /* prefill: persistent workers W >= 1; one CTA
                               runs one worker                              */
  int32_t schedule;         /* SA_SCHED_*                                   */
  int32_t group_shared;     /* prefill: 0 = one block list per query head;
                               1 = one list per KV group (GQA-group-shared
                               selection): the G heads of a group share the
                               blocks chosen on their summed scores.  Budgets
                               are Max-Min shifted between the KV groups, each
                               group demanding its most demanding head's
                               blocks, so the total stays Hq*k_uniform.
                               Must be 0 for decode.  (Fluxion, "Componenti di
                               Sistema": GQA access modelled per group.)     */
  const int32_t* granularity; /* decode: [Hq] tokens per selection block of each
                               retrieval head: a multiple of 16 that divides L,
                               with L / g <= 4096, at most 8 distinct sizes;
                               NULL = B for every head.
                               Streaming heads' entries are ignored (they keep
                               blocks of B).  Must be NULL for prefill.
                               ("Riepilogo Tecnico: Fluxion", "Intuizioni
                               Chiave" 2: block size and budget chosen per
                               retrieval head.)                              */
  const int32_t* head_budget; /* decode: [Hq] blocks each retrieval head keeps,
                               at its own block size, >= k_min (capped at its
                               block count); NULL = k_uniform.  Must be NULL
                               for prefill.                                   */
  int32_t share_kv;         /* prefill, group-shared plans with an even G: 1 =
                               the two heads of a head pair run on one K/V
                               block load (items are head pairs, see the
                               schedule below); 0 = one query head per item,
                               the pair's shared blocks then meet in L2.
                               Must be 0 otherwise.                           */
} sa_plan_params;

typedef struct sa_plan sa_plan;

/* Text for a status code (static storage; never NULL). */
const char* sa_status_string(sa_status status);

/*
 * sparse_attn_plan -- host only, no CUDA call.
 * Budgets: start every head at k_uniform; while the head with the largest
 * surplus k_h - d_h among heads above k_min exceeds the head with the
 * smallest surplus among heads below nb by more than one, move one block
 * from the first to the second (ties: lowest head).  The total is conserved.
 * Schedule (prefill): item (h, i) has id h*nb+i and cost min(k_h, i+1)
 * blocks; LPT walks items by cost descending (ties: lower id) and gives each
 * to the least-loaded worker (ties: lowest worker); LPT_GROUPED walks KV
 * group by KV group, cost descending inside a group, ties by query block
 * then head; HEAD_ORDER gives worker
 * w the contiguous id range [w*N/W, (w+1)*N/W).  Plans with share_kv = 1
 * schedule head pairs instead: item (p, i) has id p*nb+i, covers heads 2p and
 * 2p+1, and costs 2*min(k_p, i+1) blocks (G/2 pairs per KV group).
 * Decode: retrieval heads keep k_uniform blocks (or head_budget[h] blocks of
 * granularity[h] tokens), streaming heads block 0 plus the last window_blocks
 * blocks of B; no schedule is built.
 * On success *out owns a new plan (free with sparse_attn_plan_destroy).
 * Errors: INVALID_ARG (null shp/params/out, bad enum, k_min < 2, k_uniform
 * out of [k_min, max(nb, k_min)], W < 1, negative demand, a decode-only field
 * given for prefill, a bad granularity or a head budget < k_min), SHAPE,
 * UNSUPPORTED, NO_MEMORY.  *out is left untouched on error.
 */
sa_status sparse_attn_plan(const sa_shape* shp, const sa_plan_params* params,
                           sa_plan** out);

/*
 * Sizes of a plan: workers W, items N (Hq*nb prefill, Bt*Hq decode; Hq/2*nb
 * for a plan with share_kv = 1, where an item is a head pair, see
 * sparse_attn_plan), the
 * idx row stride kmax it needs (max over heads of the blocks one row keeps),
 * the total of all item costs in blocks, and the schedule's makespan (the
 * largest worker load, in blocks).  Any output pointer may be NULL.
 */
sa_status sparse_attn_plan_info(const sa_plan* plan, int32_t* num_workers,
                                int32_t* num_items, int32_t* kmax,
                                int64_t* total_blocks, int64_t* makespan);

/*
 * Decode plans: the block sizes their retrieval heads select at.
 * num_sizes, sizes[0..num_sizes) (ascending, at most 8 entries are written):
 *   the distinct block sizes of the retrieval heads (B when the plan has no
 *   granularity; none when every head streams);
 * kcache_floats: floats of the pooled key caches those sizes need together,
 *   sum over sizes g of Bt*Hkv*(L/g)*d (see sparse_attn_pool_kcache_plan);
 * score_stride: the row stride of decode scores, L / sizes[0] (nb when there
 *   are no retrieval heads).  Any output may be NULL.
 * Errors: INVALID_ARG (NULL plan, prefill plan).
 */
sa_status sparse_attn_plan_decode_layout(const sa_plan* plan, int32_t* num_sizes,
                                         int32_t* sizes, int64_t* kcache_floats,
                                         int32_t* score_stride);

/*
 * Copy a plan's contents to host arrays (any may be NULL):
 * budgets [Hq]; wptr [W+1] CSR offsets; items [N] item ids in each worker's
 * processing order; loads [W] per-worker cost in blocks.  Decode plans have
 * no schedule (W = 0): wptr gets {0}.
 */
sa_status sparse_attn_plan_get(const sa_plan* plan, int32_t* budgets,
                               int32_t* wptr, int32_t* items, int64_t* loads);

/*
 * Copy the budgets, head kinds and schedule to the current CUDA device
 * (device memory owned by the plan, freed by destroy).  Synchronises the
 * stream before returning so host staging can be reused.  Required before
 * sparse_attn_select / sparse_attn_forward.  Errors: INVALID_ARG, CUDA,
 * NO_MEMORY.  Calling it again re-uploads.
 */
sa_status sparse_attn_plan_upload(sa_plan* plan, sa_stream_t stream);

/* Free a plan and its device copy (NULL is a no-op). */
void sparse_attn_plan_destroy(sa_plan* plan);

/*
 * Scratch bytes sparse_attn_score needs: prefill (Hq + Hkv) * nb * d * 4
 * (pooled queries and keys, fp32) rounded up to 256; decode 0.
 */
sa_status sparse_attn_score_workspace_size(const sa_shape* shp, size_t* bytes);

/*
 * Index: pooled block scores.
 * Prefill: qbar[h,i] and kbar[g,j] are fp32 means of the B rows of each block
 *   (kept in ws); scores[h][i][j] = qbar[h,i] . kbar[h/G, j] / sqrt(d) for
 *   j <= i, fp32, layout [Hq][nb][nb]; entries with j > i are not written.
 *   q, k: bf16 Q and K.
 * Decode: k is the pooled key cache kbar (fp32 [Bt][Hkv][nb][d], see
 *   sparse_attn_pool_kcache); scores[b][h][j] = q[b,h] . kbar[b,h/G,j] /
 *   sqrt(d), layout [Bt][Hq][nb]; ws may be NULL.
 * The mean as the block summary is a reading: the pages select at block
 * granularity but do not name the summary.
 * Errors: INVALID_ARG (null pointers, ws_bytes too small), SHAPE,
 * UNSUPPORTED, CUDA (launch failure).
 */
sa_status sparse_attn_score(const sa_shape* shp, const void* q, const void* k,
                            float* scores, void* ws, size_t ws_bytes,
                            sa_stream_t stream);

/*
 * Index step for callers that cannot allocate device memory where they score
 * a layer: code whose hot path must not allocate (cudaMalloc may synchronise
 * the device and takes unbounded time), hosts that own all device memory
 * through their own pool and hand a plugin only its inputs and outputs, and
 * callers held to a memory budget fixed at start-up.  It computes exactly what
 * sparse_attn_score computes, but keeps the pooled queries and keys in a
 * fixed 32 MiB area of device memory that belongs to this library; the call
 * allocates nothing and takes no workspace.  A device reserves the area at the
 * first call on it (at library load when CUDA loads modules eagerly) and keeps
 * it until the process exits.  The pages have no counterpart of
 * this entry point; it exists for deployment only.
 *  - Limit: prefill shapes with (Hq + Hkv) * nb * d * 4 bytes <= 32 MiB (the
 *    Llama-3.1-8B 128K shape needs 20 MiB); larger ones return
 *    SA_ERR_UNSUPPORTED.  Decode shapes need no scratch and behave as
 *    sparse_attn_score.
 *  - The first call on each device looks up the area's device address with
 *    that device current, and may load the module that holds it; make that
 *    first call before any stream capture.  The address is kept for the life
 *    of the process: do not call this entry point again after cudaDeviceReset
 *    or any other teardown of the device's primary context.
 *  - All calls on a device share the area.  Each call rewrites every pooled
 *    vector it reads, so nothing has to be cleared, but calls whose execution
 *    overlaps on the GPU (other streams, other host threads) race on it:
 *    serialise them.
 * Errors: as sparse_attn_score, plus UNSUPPORTED for the size limit.
 */
sa_status sparse_attn_score_noalloc(const sa_shape* shp, const void* q, const void* k,
                                    float* scores, sa_stream_t stream);

/*
 * Select: for prefill row (h, i) keep min(k_h, i+1) blocks: 0 and i always,
 * then the highest-scoring of 1..i-1, ties to the lower index.  For decode
 * retrieval heads the row is i = nb_h - 1 with k_h the head's budget, nb_h =
 * L / granularity[h] blocks (nb without a granularity) and score rows of the
 * plan's score_stride floats (nb without a granularity); streaming heads get
 * block 0 and the last window_blocks blocks of B.  Decode rows of up to 4096
 * blocks are supported.
 * Group-shared plans (sa_plan_params.group_shared = 1, prefill): one list per
 * (KV group g, row i), chosen as above on the sum over the group's G heads of
 * their scores (the order of their mean) with the group's budget, and written
 * to the rows of all G heads.
 * Outputs: idx [rows][kmax] int32, each row ascending and padded with -1;
 * cnt [rows] int32; rows = Hq*nb (prefill, row h*nb+i) or Bt*Hq (decode,
 * row b*Hq+h).  kmax must be >= the plan's kmax (sparse_attn_plan_info).
 * Prefill rows of up to 2048 blocks are supported (nb <= 2048), else UNSUPPORTED.
 * Errors: INVALID_ARG, SHAPE (kmax too small, shape differs from the plan's),
 * UNSUPPORTED, NOT_UPLOADED, CUDA.
 */
sa_status sparse_attn_select(const sa_shape* shp, const sa_plan* plan,
                             const float* scores, int32_t* idx, int32_t* cnt,
                             int32_t kmax, sa_stream_t stream);

/*
 * Decode plans only: sparse_attn_select restricted to the rows of the heads
 * of one kind, head_kind = SA_HEAD_STREAMING or SA_HEAD_RETRIEVAL (rows b*Hq+h
 * of the other heads are left as they are).  Streaming heads keep block 0 and
 * the last window blocks whatever the scores say, so their lists can be made
 * (and attended, sparse_attn_forward_kind) on one stream while the retrieval
 * heads score and select on another: Fluxion's split into streaming and
 * retrieval heads ("Riepilogo Tecnico: Fluxion", "Intuizioni Chiave" 1) lets
 * the two kinds proceed independently.  scores may be NULL for
 * SA_HEAD_STREAMING.  A kind with no head returns SA_OK and launches nothing.
 * Errors: as sparse_attn_select, plus INVALID_ARG for a prefill plan or an
 * unknown kind.
 */
sa_status sparse_attn_select_kind(const sa_shape* shp, const sa_plan* plan,
                                  const float* scores, int32_t* idx, int32_t* cnt,
                                  int32_t kmax, int32_t head_kind, sa_stream_t stream);

/*
 * Decode plans without per-head block sizes: the Index and Select steps of
 * the retrieval heads in one launch (Spin's Index / Select split, "Abstracción
 * de Partición Unificada"; the retrieval rows of "Riepilogo Tecnico: Fluxion",
 * "Intuizioni Chiave" 1 and 2).  The results are those of sparse_attn_score
 * followed by sparse_attn_select_kind(SA_HEAD_RETRIEVAL), bit for bit, but the
 * scores need not leave the chip: one thread-block cluster per (sequence, KV
 * group) scores the group's pooled keys in shared memory and selects from
 * there, so the selection does not wait for a second launch.
 *  - q: bf16 [Bt][Hq][d]; kbar: the pooled key cache (fp32 [Bt][Hkv][nb][d],
 *    sparse_attn_pool_kcache).
 *  - scores: fp32 [Bt][Hq][nb], or NULL.  When given, the rows of the
 *    retrieval heads receive their scores; other rows are left as they are.
 *  - idx [Bt*Hq][kmax], cnt [Bt*Hq]: the rows b*Hq+h of the retrieval heads,
 *    as sparse_attn_select writes them; the streaming heads' rows are left as
 *    they are (sparse_attn_select_kind(SA_HEAD_STREAMING) writes them).
 * All pointers are device pointers, q, kbar and scores 16-byte aligned.  A
 * plan with no retrieval head returns SA_OK and launches nothing.
 * Errors: INVALID_ARG (NULL pointers, misalignment, prefill plan), SHAPE
 * (shape differs from the plan's, kmax too small), NOT_UPLOADED, UNSUPPORTED
 * (a plan with per-head block sizes, d != 128, Hq/Hkv > 16, nb > 4096), CUDA.
 */
sa_status sparse_attn_score_select(const sa_shape* shp, const sa_plan* plan, const void* q,
                                   const float* kbar, float* scores, int32_t* idx,
                                   int32_t* cnt, int32_t kmax, sa_stream_t stream);

/*
 * Decode plans without per-head block sizes, block size 32: the whole decode
 * step in one launch.  The results are those of sparse_attn_score_select,
 * sparse_attn_select_kind(SA_HEAD_STREAMING) and sparse_attn_forward, bit for
 * bit: scores (retrieval rows, when scores is not NULL), idx and cnt (every
 * row), o and lse (every row).  One thread-block cluster per (sequence, KV
 * group) scores and selects the group's retrieval heads as
 * sparse_attn_score_select does; the warpgroup that selected a head then
 * attends it at once, and the group's streaming heads (block 0 and the last
 * window_blocks blocks, "Riepilogo Tecnico: Fluxion", "Intuizioni Chiave" 2)
 * are attended by the cluster's other warpgroups.  No head waits for a
 * second launch, so attention reads overlap the other heads' selection.
 *  - q: bf16 [Bt][Hq][128]; kbar: the pooled key cache (fp32
 *    [Bt][Hkv][nb][128], sparse_attn_pool_kcache); k, v: bf16
 *    [Bt][Hkv][L][128].
 *  - scores: fp32 [Bt][Hq][nb] or NULL; idx [Bt*Hq][kmax], cnt [Bt*Hq]: as
 *    sparse_attn_select writes them.
 *  - o [Bt*Hq][128] in o_dtype (SA_DTYPE_BF16 or SA_DTYPE_F32); lse
 *    (nullable) [Bt*Hq]; dev_status: as sparse_attn_forward (an out-of-range
 *    count or index is flagged, a copy wait that passes the limit of
 *    sparse_attn_set_wait_limit sets SA_DEV_TIMEOUT).
 * All pointers are device pointers; q, kbar, k, v, o and scores 16-byte
 * aligned.  The launch holds up to ~110 KB of shared memory per CTA (two CTAs
 * per SM at the common shapes).
 * Errors: INVALID_ARG (NULL pointers, misalignment, o_dtype, prefill plan),
 * SHAPE (shape differs from the plan's, kmax too small), NOT_UPLOADED,
 * UNSUPPORTED (per-head block sizes, block size other than 32, d != 128,
 * Hq/Hkv > 16, nb > 4096), CUDA.
 */
sa_status sparse_attn_decode_step(const sa_shape* shp, const sa_plan* plan, const void* q,
                                  const float* kbar, const void* k, const void* v, float* scores,
                                  int32_t* idx, int32_t* cnt, int32_t kmax, void* o,
                                  int32_t o_dtype, float* lse, int32_t* dev_status,
                                  sa_stream_t stream);

/*
 * Top-p selection, the data-dependent alternative the S-HPLB pages compare
 * against (Italian summary, "Sparsita' Eterogenea": an adaptive top-p budget
 * fixes accuracy but makes every head's work different).  Prefill only.
 * Row (h, i): block probabilities are the softmax of the row's pooled scores
 * over j <= i; the row keeps blocks 0 and i, then blocks of 1..i-1 by score
 * (ties: lower index) until the kept probability reaches p (p >= 1 keeps the
 * row's all blocks, p <= 0 only 0 and i).  Probabilities are summed in 64-bit
 * fixed point (2^-32 of the row's total), so results are reproducible.
 * Outputs as sparse_attn_select; kmax must be >= nb since a row may keep all
 * its blocks.  The plan's budgets are not used; its schedule assumes them, so
 * rebuild it from cnt (sparse_attn_plan_rebuild) before the forward.
 * Errors: INVALID_ARG (NULL, NaN p, decode), SHAPE, UNSUPPORTED (nb > 2048),
 * NOT_UPLOADED, CUDA.
 */
sa_status sparse_attn_select_topp(const sa_shape* shp, const sa_plan* plan,
                                  const float* scores, float p, int32_t* idx,
                                  int32_t* cnt, int32_t kmax, sa_stream_t stream);

/*
 * Rebuild a prefill plan's device schedule from device block counts
 * cnt [Hq*nb] (e.g. from sparse_attn_select_topp), on the GPU: LPT with item
 * cost cnt[item] -- items by cost descending (ties: lower id), each to the
 * least-loaded worker (ties: lowest worker) -- written over the plan's device
 * wptr / items, which sparse_attn_forward reads.  Each worker's items are
 * listed in ascending item id (head-major), so that CTAs running at the same
 * time tend to read the same KV head.  One single-CTA kernel on `stream`
 * (about 148 KB of shared memory); the first call allocates 3*N int32 of
 * scratch, owned by the plan.  Counts outside [0, 2048] are clamped
 * to it.  The host copy of the schedule (sparse_attn_plan_get / _info) is not
 * changed.  Up to 256 workers, nb <= 2048 and N = Hq*nb <= 2^19 items, else
 * UNSUPPORTED.
 * Errors: INVALID_ARG (NULL, decode plan), NOT_UPLOADED, UNSUPPORTED, CUDA.
 */
sa_status sparse_attn_plan_rebuild(sa_plan* plan, const int32_t* cnt, sa_stream_t stream);

/*
 * Copy the plan's device schedule (wptr [W+1], items [N]) into caller
 * buffers, host or device (cudaMemcpyDefault), asynchronously on `stream`.
 * Errors: INVALID_ARG, NOT_UPLOADED, CUDA.
 */
sa_status sparse_attn_plan_device_schedule(const sa_plan* plan, int32_t* wptr,
                                           int32_t* items, sa_stream_t stream);

/*
 * Decode plans only: sparse_attn_forward restricted to the rows (b, h) of the
 * heads of one kind (see sparse_attn_select_kind); the other rows of o and lse
 * are not written.  The plan is required and must be uploaded.  A kind with no
 * head returns SA_OK and launches nothing.
 * Errors: as sparse_attn_forward, plus INVALID_ARG for a prefill plan or an
 * unknown kind.
 */
sa_status sparse_attn_forward_kind(const sa_shape* shp, const sa_plan* plan,
                                   const void* q, const void* k, const void* v,
                                   const int32_t* idx, const int32_t* cnt, int32_t kmax,
                                   void* o, int32_t o_dtype, float* lse,
                                   int32_t* dev_status, int32_t head_kind,
                                   sa_stream_t stream);

/*
 * Watchdog limit of the forward kernels: every wait of one role on another
 * in the prefill kernel (a copy landing, a tensor-core result, a softmax
 * step), and every wait for a copy in the decode kernel, gives up after `ns`
 * nanoseconds of GPU global time, for launches made after this call by any
 * thread of the process.  0 restores the default, 4 s.
 * A CTA whose wait runs out ORs SA_DEV_TIMEOUT into dev_status, stops every
 * role of the CTA, lets the copies and tensor-core operations it already
 * issued complete (those waits keep the 4 s limit), frees its tensor memory
 * and exits: the launch ends with invalid output but the context stays
 * usable.  Callers that would rather see an error than a stalled stream set
 * a limit near their own deadline; short limits also let a test take this
 * path on purpose.  Returns SA_OK.
 */
sa_status sparse_attn_set_wait_limit(uint64_t ns);

/*
 * Attention over the selected blocks.
 * Prefill: o[h, t] = sum_u softmax_u(q[h,t] . k[g,u] / sqrt(d)) v[g,u] over
 *   the keys u of the blocks idx[h*nb+i][0..cnt) with u <= t (only the
 *   diagonal block is partly masked); online softmax in fp32; the bf16
 *   probabilities fed to the P.V product also form the normaliser, so each
 *   output row is a convex combination of value rows.
 *   Runs as a persistent kernel: one CTA per plan worker, walking that
 *   worker's items in order (sm_103a: TMA loads, tcgen05 MMAs into TMEM).
 * Decode: o[b,h] over the blocks of row b*Hq+h, block j of head h covering
 *   tokens [j*g_h, (j+1)*g_h) with g_h = granularity[h] of the plan (B when
 *   the plan has none, or when plan is NULL).
 * o_dtype: SA_DTYPE_BF16 (round to nearest even) or SA_DTYPE_F32.
 * lse (nullable): natural-log sum of exponentials per query row, fp32,
 *   [Hq][S] (prefill) or [Bt][Hq] (decode).
 * dev_status: device int32 the kernels OR SA_DEV_* bits into (not cleared by
 *   the library); an out-of-range index or count is clamped and flagged, never
 *   dereferenced.
 * Errors: INVALID_ARG, SHAPE, UNSUPPORTED, NOT_UPLOADED, CUDA.
 */
sa_status sparse_attn_forward(const sa_shape* shp, const sa_plan* plan,
                              const void* q, const void* k, const void* v,
                              const int32_t* idx, const int32_t* cnt,
                              int32_t kmax, void* o, int32_t o_dtype, float* lse,
                              int32_t* dev_status, sa_stream_t stream);

/*
 * Decode: build the pooled key cache kbar[b][g][j] = mean of the B keys of
 * block j (fp32, [Bt][Hkv][nb][d]) from K [Bt][Hkv][L][d].  Done once per
 * cache; the retrieval heads' scores read it.
 * Errors: INVALID_ARG, SHAPE, UNSUPPORTED, CUDA.
 */
sa_status sparse_attn_pool_kcache(const sa_shape* shp, const void* k,
                                  float* kbar, sa_stream_t stream);

/*
 * Decode with per-head block sizes: the pooled key caches of every size the
 * plan's retrieval heads use, one after the other in ascending size, each
 * fp32 [Bt][Hkv][L/g][d] (the mean of the g keys of each block), into kbar_all
 * (sparse_attn_plan_decode_layout gives the total floats).  Once per cache.
 * Errors: INVALID_ARG (NULL, prefill plan), SHAPE (shape differs from the
 * plan's), UNSUPPORTED, CUDA.
 */
sa_status sparse_attn_pool_kcache_plan(const sa_shape* shp, const sa_plan* plan,
                                       const void* k, float* kbar_all,
                                       sa_stream_t stream);

/*
 * Decode with per-head block sizes: scores[b][h][j] = q[b,h] . kbar_g[b,h/G,j]
 * / sqrt(d) for each retrieval head h at its block size g = granularity[h],
 * j < L/g, rows of the plan's score_stride floats ([Bt][Hq][score_stride]);
 * streaming heads' rows are not written.  One pass per block size; a KV group
 * none of whose heads uses a size does not read that size's cache.
 * Errors: INVALID_ARG, SHAPE, UNSUPPORTED, CUDA.
 */
sa_status sparse_attn_score_plan(const sa_shape* shp, const sa_plan* plan,
                                 const void* q, const float* kbar_all,
                                 float* scores, sa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPARSE_ATTN_H */
