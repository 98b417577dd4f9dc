/*
 * ra.h - C ABI of a GB300 (sm_103a) library for the chunked forward pass of
 * ring attention: exact softmax attention computed one key/value chunk at a
 * time and combined with the online-softmax merge rule.
 *
 * Sources (web pages, cited by title and section):
 *   [EX]   ring-attention exercise "systems-distributed-ring-attention-online-
 *          softmax": task statement and hints.
 *   [BLOG] "Ring Attention: Distributed Reads with Online Softmax".
 *   [GLOS] glossary entry "ring attention".
 *   [IRIS] pull request "Support ring attention" (IRIS, Triton, MI300X),
 *          commit messages.
 *
 * Common conventions
 * ------------------
 * - Every pointer passed to a compute entry point is a DEVICE pointer owned
 *   by the caller (ra_ring_attention_host alone takes host pointers); the
 *   library never frees or retains it. The only device memory the library
 *   itself allocates is the per-call scratch of ra_ring_attention and the
 *   device copies of ra_ring_attention_host, stream-ordered, from one library
 *   memory pool per device. Descriptor structs are read on the host during
 *   the call only.
 * - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *   stream). A returned RA_OK means the work was validated and enqueued.
 * - Every argument is validated before anything is enqueued. On any non-OK
 *   status nothing was launched and no output was written;
 *   ra_last_error() then returns a message for the calling thread.
 * - Tensors are [batch, head, row, head_dim] with head_dim contiguous and the
 *   other three axes given by element strides (ra_strides).
 * - Query head h reads key/value head h / (Hq / Hkv) (grouped heads).
 * - Scores are s = scale * <q, k>. The row max m is returned in those scaled,
 *   natural-log units and l = sum exp(s - m) over the keys the row may see.
 * - Causal masking uses GLOBAL positions ([BLOG] "Causal masks depend on
 *   global positions"): key j is visible to query i iff pos(j) <= pos(i).
 *   Positions are described per chunk / query segment by spans.
 * - Packed documents (optional, ra_problem.doc_bounds): several variable-
 *   length sequences share one position range; a query sees only the keys of
 *   its own document, causal or not. The pages do not discuss packing: this
 *   is the plainest extension of the global-position mask.
 * - A row that sees no key gets O = 0 (or u = 0), l = 0, m = -inf.
 * - dtype RA_BF16: Q, K, V and O are bfloat16; products are accumulated in
 *   fp32 on the tensor cores; head_dim must be 64, 96 or 128.
 *   dtype RA_F32: everything is fp32 on CUDA cores (no TF32); head_dim
 *   1..128.
 */
#ifndef RA_H_
#define RA_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RA_OK = 0,
  RA_ERR_INVALID = 1,      /* bad argument: nothing was launched            */
  RA_ERR_UNSUPPORTED = 2,  /* valid but outside what this build handles      */
  RA_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed              */
  RA_ERR_TIMEOUT = 4       /* a kernel gave up waiting (see ra_device_status) */
} ra_status;

typedef enum { RA_F32 = 0, RA_BF16 = 1 } ra_dtype;

#define RA_MAX_SPANS 4
#define RA_MAX_DOCS 512

/* Rows [r, r + len) of a chunk / segment have global positions
 * pos0, pos0 + step, ..., pos0 + (len - 1) * step.  step >= 1. */
typedef struct {
  int64_t len;
  int64_t pos0;
  int64_t step;
} ra_span;

/* Positions of consecutive rows: the spans are concatenated in order and their
 * lengths add up to the owner's row count. One span describes a contiguous
 * shard; two describe a zigzag (early block + late block) shard; a span with
 * step P describes a striped shard. Positions must lie in [0, 2^31 - 1). */
typedef struct {
  int32_t nspan;            /* 1..RA_MAX_SPANS */
  int32_t reserved;         /* must be 0 */
  ra_span span[RA_MAX_SPANS];
} ra_positions;

typedef struct {
  int64_t batch, head, row; /* element strides; head_dim is contiguous */
} ra_strides;

/* One key/value chunk ("shard" on the pages). K and V are [B, Hkv, len, D]. */
typedef struct {
  const void* k;
  const void* v;
  int64_t len;              /* rows in this chunk (0 = empty chunk, skipped) */
  ra_strides k_strides;
  ra_strides v_strides;
  ra_positions pos;         /* global position of each row */
} ra_kv_chunk;

/* One query segment: the next `len` rows of Q (segments tile Q's rows in
 * order). With as many segments as chunks, segment r plays device r of the
 * ring and visits chunks r, r-1, ..., r+1 (mod P): at ring step s it holds the
 * chunk that started on device r - s ([BLOG] "Partition the sequence across
 * devices"; [GLOS] algorithm steps (1)-(5)). Otherwise every segment visits
 * the chunks in index order. The result does not depend on the order beyond
 * rounding. */
typedef struct {
  int64_t len;
  ra_positions pos;
} ra_q_segment;

typedef struct {
  int64_t B, Hq, Hkv, D;
  int64_t Sq;               /* query rows (sum of the segment lengths) */
  int32_t dtype;            /* ra_dtype of Q, K, V and O */
  int32_t causal;           /* 0 or 1 */
  float scale;              /* score scale; <= 0 selects 1/sqrt(D) */
  int32_t o_fp32;           /* 1: write O in fp32 even for bf16 inputs; 0: O has
                               the input dtype. (A bf16 O carries its own
                               rounding of up to 2^-9 relative.) */
  ra_strides q_strides;     /* Q: [B, Hq, Sq, D] */
  ra_strides o_strides;     /* O (ring) or u (chunk stats): [B, Hq, Sq, D] */
  /* Packed documents. n_docs = 0: one document holds every position and
     doc_bounds is ignored. n_docs in 1..RA_MAX_DOCS: doc_bounds is a HOST
     array of n_docs + 1 strictly increasing positions b_0 < ... < b_n (read
     during the call only); document d holds positions [b_d, b_{d+1}) and key
     j is visible to query i only if both lie in the same document (and, when
     causal, pos(j) <= pos(i)). Every query and key position must lie in
     [b_0, b_n) (else RA_ERR_INVALID). The same documents apply to every batch
     element and head. */
  const int64_t* doc_bounds;
  int32_t n_docs;
  int32_t reserved_docs;    /* must be 0 */
} ra_problem;

/*
 * ra_chunk_stats - statistics of ONE key/value chunk for every query row,
 * computed as if that chunk were the only one ([EX] task statement:
 * attention_chunk_stats returns chunk_output, chunk_sum, chunk_max; [EX] hint
 * 1: the max-subtraction of scaled dot-product attention, with numerator and
 * denominator returned separately).
 *
 *   u [B, Hq, Sq, D] fp32 (problem->o_strides): sum_j exp(s_ij - m_i) v_j
 *   l [B, Hq, Sq]    fp32 contiguous:           sum_j exp(s_ij - m_i)
 *   m [B, Hq, Sq]    fp32 contiguous:           max_j s_ij  (-inf if none)
 *
 * q is [B, Hq, Sq, D] of problem->dtype; segs give the query positions
 * (their ring roles do not matter here).
 */
ra_status ra_chunk_stats(const ra_problem* problem, const void* q,
                         const ra_q_segment* segs, int32_t nsegs,
                         const ra_kv_chunk* chunk,
                         float* u, float* l, float* m, void* stream);

/*
 * ra_merge_stats - the online-softmax merge of two sets of statistics, in
 * place into the accumulator ([EX] task statement and hint 2; [BLOG] "Do not
 * average independently normalized shard outputs"):
 *
 *   m' = max(m_acc, m_new);  a = exp(m_acc - m'), b = exp(m_new - m')
 *   u_acc = a u_acc + b u_new;  l_acc = a l_acc + b l_new;  m_acc = m'
 *
 * A side with m = -inf contributes nothing (a or b taken as 0). All arrays
 * are fp32 and contiguous: u [rows, D], l and m [rows]. The _new arrays may
 * not overlap the _acc arrays unless identical.
 */
ra_status ra_merge_stats(int64_t rows, int64_t D,
                         float* u_acc, float* l_acc, float* m_acc,
                         const float* u_new, const float* l_new,
                         const float* m_new, void* stream);

/*
 * ra_merge_lse - the same merge in log-sum-exp form, for composing with
 * kernels that return a normalised output and its row log-sum-exp ([GLOS]
 * "Online softmax": outputs of different key/value blocks are combined with
 * the log-sum-exp trick). In place into the accumulator:
 *
 *   lse' = log(exp(lse_acc) + exp(lse_new))
 *   o_acc = exp(lse_acc - lse') o_acc + exp(lse_new - lse') o_new
 *
 * lse is the natural log of a row's softmax denominator in the units of the
 * scaled scores (lse = m + log(l)); a side with lse = -inf weighs nothing and
 * two such sides give o = 0, lse = -inf. fp32, contiguous: o [rows, D], lse
 * [rows]. The _new arrays may not overlap the _acc arrays unless identical.
 */
ra_status ra_merge_lse(int64_t rows, int64_t D, float* o_acc, float* lse_acc,
                       const float* o_new, const float* lse_new, void* stream);

/*
 * ra_stats_to_lse - lse = m + log(l) per row (-inf where l = 0), from the
 * m, l of ra_ring_attention or ra_chunk_stats. fp32, contiguous [rows]; lse
 * may alias m or l.
 */
ra_status ra_stats_to_lse(int64_t rows, const float* m, const float* l, float* lse,
                          void* stream);

/*
 * ra_ring_attention - the whole chunked forward pass in one persistent
 * kernel: each query tile walks the key/value chunks in its segment's ring
 * order, keeping m, l and the output accumulator on chip across all chunks,
 * and finally writes O = u / l ([EX] task statement: ring_attention must equal
 * ordinary attention over the concatenated key/value sequence for any
 * chunking; [BLOG] "A simple forward schedule"; [GLOS] algorithm (1)-(6)).
 *
 *   O [B, Hq, Sq, D] of problem->dtype, or fp32 if problem->o_fp32
 *     (problem->o_strides)
 *   m [B, Hq, Sq] fp32 contiguous: the true row max of scaled scores
 *   l [B, Hq, Sq] fp32 contiguous: sum exp(s - m) over visible keys
 *
 * Causal key/value tiles that lie entirely in a query tile's future are
 * skipped; only tiles that straddle the diagonal are masked elementwise.
 * When the last rounds of work are split across CTAs (bf16 path), the call
 * allocates a scratch buffer of up to about 21 MB from the library's memory
 * pool on `stream` (cudaMallocFromPoolAsync) and frees it with cudaFreeAsync
 * on the same stream. A bf16 problem with more than 32 chunks, 64 key spans or
 * 64 query spans keeps its chunk tables (tensor maps, spans) in device
 * memory: a further ~256 bytes per chunk from the same allocation, filled by
 * one copy from the host on `stream`.
 * Limits of this build (RA_ERR_UNSUPPORTED beyond them): bf16 at most 4096
 * chunks, 8192 key spans and 8192 query spans; fp32 at most 256 chunks, 320
 * key spans and 64 query spans.
 */
ra_status ra_ring_attention(const ra_problem* problem, const void* q,
                            const ra_q_segment* segs, int32_t nsegs,
                            const ra_kv_chunk* chunks, int32_t nchunks,
                            void* o, float* m, float* l, void* stream);

/* Gradient outputs of one key/value chunk (ra_ring_attention_bwd): fp32,
 * dense [B, Hkv, len, D], caller-owned device memory. */
typedef struct {
  float* dk;
  float* dv;
} ra_kv_grad;

/*
 * ra_ring_attention_bwd - gradients of ra_ring_attention's O with respect to
 * Q and to the K and V of every chunk, given dO ([BLOG] "Backward must
 * aggregate shared dependencies": a query row's gradient reaches every chunk
 * it attended to; each chunk's dK, dV sum the contributions of all query rows
 * for the chunk's owner; probability tiles are recomputed with the forward's
 * scale and masks):
 *
 *   P = softmax of the visible scaled scores (fixed by the forward's m, l)
 *   dV = P^T dO;  dS = P * (dO V^T - rowsum(dO * O));  dQ = scale dS K;
 *   dK = scale dS^T Q;  with grouped heads, K/V head g sums over its query heads.
 *
 * problem, q, segs, chunks: exactly as given to ra_ring_attention (same
 * positions, mask, scale). o, m, l: that call's outputs (o bf16, or fp32 when
 * problem->o_fp32, with problem->o_strides). dout: bf16 [B, Hq, Sq, D] with
 * problem->o_strides (multiples of 8 elements). Outputs, fp32 and dense: dq
 * [B, Hq, Sq, D]; grads[k].dk, grads[k].dv [B, Hkv, len_k, D] for every chunk
 * with len_k > 0 (all zero when no query sees the chunk). The call takes a
 * scratch buffer from the library's memory pool on `stream` and frees it
 * again: two floats per query row and 9232 bytes per 128-row query tile and
 * query head (the key/value CTAs' per-column data, about 72 bytes per query
 * row).
 * bf16 inputs only (RA_ERR_UNSUPPORTED for RA_F32); head_dim 64, 96 or 128; the
 * chunk and span limits of ra_ring_attention's bf16 path.
 */
ra_status ra_ring_attention_bwd(const ra_problem* problem, const void* q,
                                const ra_q_segment* segs, int32_t nsegs,
                                const ra_kv_chunk* chunks, int32_t nchunks,
                                const void* o, const void* dout, const float* m,
                                const float* l, float* dq, const ra_kv_grad* grads,
                                void* stream);

/*
 * ra_ring_attention_noalloc - ra_ring_attention for callers that must not
 * allocate device memory. (The pages have no counterpart: this is a
 * deployment variant of the same kernel.)
 *
 * ra_ring_attention may allocate a per-call scratch buffer (stream-ordered,
 * freed again at the end of the call) when it splits a work unit across CTAs.
 * Some callers cannot allow that: a process whose device memory is entirely
 * reserved by another allocator (for example a framework's caching pool
 * sized to the whole GPU), where a foreign allocation fails or fragments
 * memory; or a deployment that must keep its footprint fixed after start-up
 * and may not allocate on the request path. This entry point computes the
 * same results with the same kernel, but takes its scratch from one fixed
 * array of RA_NOALLOC_SCRATCH_BYTES in the library's device image; every GPU
 * that loads the library holds that array until the process exits. It calls
 * no cudaMalloc, cudaFree or other allocating routine.
 *
 * - The first call on a device looks up the array's device address (once per
 *   device, with that device current). Make that first call before any
 *   stream capture.
 * - All calls share the array and it keeps the last call's contents; the
 *   parts that must start cleared are cleared by each call on its stream.
 *   Calls whose kernels overlap on the GPU (other streams, other threads)
 *   race on the array: serialise them.
 * - The array also holds the device-resident chunk tables of problems with
 *   more than 32 chunks or 64 spans (copied in on `stream`). A problem whose
 *   split scratch and chunk tables need more than the array holds is
 *   rejected with RA_ERR_UNSUPPORTED before anything is launched.
 * Arguments, layouts and results are those of ra_ring_attention.
 */
#define RA_NOALLOC_SCRATCH_BYTES (24u << 20)
ra_status ra_ring_attention_noalloc(const ra_problem* problem, const void* q,
                                    const ra_q_segment* segs, int32_t nsegs,
                                    const ra_kv_chunk* chunks, int32_t nchunks,
                                    void* o, float* m, float* l, void* stream);

/*
 * ra_ring_attention_host - ra_ring_attention with every input and output in
 * HOST memory. (The pages have no counterpart: this is the end-to-end form of
 * the same pass, for callers whose tensors live on the host.)
 *
 * All work is stream-ordered on `stream`: the library takes device buffers
 * for Q, the chunks, O, m and l from its memory pool, copies the inputs in
 * (issued only after the problem has been validated and planned), runs the
 * kernel of ra_ring_attention, copies O, m and l out and releases the
 * buffers. The call returns once all of that is enqueued. Tensors that lie
 * back to back inside one pinned host allocation (q, then the k of every
 * chunk, then the v of every chunk; o, m, l) are copied with one
 * cudaMemcpyAsync per run, others with one each. The host buffers must stay
 * valid and unchanged until `stream` has passed this call
 * (cudaStreamSynchronize, an event); page-locked (pinned) host memory gives
 * full copy bandwidth and truly asynchronous copies. Calls on different
 * streams overlap one call's copies with another call's kernel (no call
 * waits for another stream's release of pool memory).
 *
 * Arguments, positions and results are those of ra_ring_attention, with two
 * differences: every pointer (q, chunks[k].k, chunks[k].v, o, m, l) is a host
 * pointer, and every tensor must be dense: q and o as [B, Hq, Sq, D], the k
 * and v of chunk k as [B, Hkv, len_k, D] (strides of axes with extent 1 are
 * ignored); RA_ERR_INVALID otherwise. The pool keeps up to 4 GiB mapped
 * between calls.
 */
ra_status ra_ring_attention_host(const ra_problem* problem, const void* q,
                                 const ra_q_segment* segs, int32_t nsegs,
                                 const ra_kv_chunk* chunks, int32_t nchunks,
                                 void* o, float* m, float* l, void* stream);

/*
 * ra_segment_work - host-only bookkeeping for comparing sequence layouts
 * ([BLOG] "Causal masks depend on global positions": contiguous causal
 * sharding is imbalanced, paired early/late chunks even it out; [GLOS]
 * "Variants (1) striped attention"). For each query segment r:
 *   pairs[r] = number of (query row, key row) pairs of that segment that the
 *              causal mask leaves visible, for one (batch, head);
 *   tiles[r] = number of (128-row query tile, 128-row key tile) products the
 *              bf16 kernel schedules for it after skipping dead tiles.
 * Either output may be NULL. No device work.
 */
ra_status ra_segment_work(const ra_problem* problem,
                          const ra_q_segment* segs, int32_t nsegs,
                          const ra_kv_chunk* chunks, int32_t nchunks,
                          int64_t* pairs, int64_t* tiles);

/*
 * ra_device_status - waits for `stream`, then reports whether any kernel of
 * this library gave up on a bounded wait since the last call (RA_ERR_TIMEOUT;
 * the flag is cleared) or whether the stream holds a CUDA error
 * (RA_ERR_CUDA). Kernels never spin forever: every wait on the chip has a time
 * budget after which the kernel records the timeout and exits cleanly.
 */
ra_status ra_device_status(void* stream);

/* Message for the calling thread's last non-OK status ("" if none). */
const char* ra_last_error(void);

/* ABI version of this header: 10000 * major + 100 * minor + patch. */
int32_t ra_version(void);

#define RA_VERSION 101

#ifdef __cplusplus
}
#endif

#endif /* RA_H_ */
