// Internal launch plans of the ring-attention kernels.
//
// A plan is built on the host from the caller's descriptors and passed to a
// kernel BY VALUE as a __grid_constant__ parameter (at most 32 KB), so a call
// needs no device allocation and no host-to-device copy besides the launch.
// Rows and positions are 32-bit here; the host validates that they fit.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace ra {

// Rows [row0, row0 + len) of Q have global positions pos0 + step * (i - row0).
// `seg` is the query segment the rows belong to (its ring role).
struct QPiece {
  int32_t row0, len, pos0, step, seg;
};

// One monotone span of a key/value chunk, the unit the kernels iterate over:
// rows [row0, row0 + len) of chunk `chunk`, positions pos0 + step * (i - row0).
struct KvSeg {
  int32_t chunk, row0, len, pos0, step, ntiles;  // ntiles: 128-row tiles
};

constexpr int kMaxQPieces = 64;
constexpr int kMaxDocs = 512;

#if defined(__CUDACC__)
// Loads of span records from device-resident tables (read-only path). The
// kernels read a plan's own tables directly and a device-resident copy only
// through these, in separate branches: one access that might point to either
// would become a generic load, which costs a memory round trip even for the
// plan's own arrays.
__device__ __forceinline__ QPiece ld_qpiece(const QPiece* q) {
  QPiece r;
  r.row0 = __ldg(&q->row0);
  r.len = __ldg(&q->len);
  r.pos0 = __ldg(&q->pos0);
  r.step = __ldg(&q->step);
  r.seg = __ldg(&q->seg);
  return r;
}
__device__ __forceinline__ KvSeg ld_kvseg(const KvSeg* k) {
  KvSeg r;
  r.chunk = __ldg(&k->chunk);
  r.row0 = __ldg(&k->row0);
  r.len = __ldg(&k->len);
  r.pos0 = __ldg(&k->pos0);
  r.step = __ldg(&k->step);
  r.ntiles = __ldg(&k->ntiles);
  return r;
}
#endif

#if defined(__CUDACC__)
#define RA_HD __host__ __device__ __forceinline__
#else
#define RA_HD inline
#endif

// Packed documents: a plan with n_docs > 0 holds boundaries b_0 < ... < b_n
// (doc_bounds[0 .. n_docs]); document d is the position range [b_d, b_{d+1})
// and a query sees only keys of its own document. The window of a query at
// position pos is the key positions [lo, hi] it may see: its document (all
// positions when there are no documents), cut at pos itself when causal.
// Every plan type below carries the same three members used here.
template <class Plan>
RA_HD void key_window(const Plan& p, int pos, int& lo, int& hi) {
  lo = 0;
  hi = p.causal ? pos : 0x7fffffff;
  if (p.n_docs > 0) {
    int a = 0, z = p.n_docs - 1;  // last d with b_d <= pos
    while (a < z) {
      const int mid = (a + z + 1) >> 1;
      if (p.doc_bounds[mid] <= pos) a = mid; else z = mid - 1;
    }
    lo = p.doc_bounds[a];
    if (!p.causal) hi = p.doc_bounds[a + 1] - 1;
  }
}

// Work unit u -> the rank of its query-tile pair in the visit order, its
// batch and its query head. Units come in blocks of pair_block pair ranks
// (the last block may be shorter); inside a block the key/value streams
// (batch, key/value head) are outermost, then the pair, then the query heads
// sharing the stream. pair_block = 1: pair-major, heads innermost.
RA_HD void unit_coords(int u, int n_qpairs, int B, int Hq, int Hkv, int pair_block, int& rank,
                       int& b, int& hq) {
  const int gq = Hq / Hkv, BH = B * Hq;
  const int blk = u / (pair_block * BH);
  const int w = u - blk * (pair_block * BH);
  const int pe = (n_qpairs - blk * pair_block) < pair_block ? (n_qpairs - blk * pair_block) : pair_block;
  const int s = w / (pe * gq), rem = w - s * (pe * gq);
  const int pi = rem / gq, j = rem - pi * gq;
  rank = blk * pair_block + pi;
  b = s / Hkv;
  hq = (s - b * Hkv) * gq + j;
}

// Tiles [tb, te) of a monotone key span (positions pos0 + step * i, len rows,
// 128-row tiles) that hold at least one position inside [lo, hi]. The host
// (work estimates) and the kernels (tile walks) share this arithmetic, so
// both count the same tiles. Positions lie in [0, 2^31 - 1), so every
// difference below fits in 31 bits; unit steps (contiguous and zigzag spans)
// need no division.
RA_HD void live_range(int pos0, int step, int len, int lo, int hi, int& tb, int& te) {
  const int nt = (len + 127) >> 7;
  if (hi < pos0 || len <= 0) {
    tb = te = 0;
    return;
  }
  const unsigned dh = static_cast<unsigned>(hi - pos0);
  const unsigned last = step == 1 ? dh : dh / static_cast<unsigned>(step);  // last row with pos <= hi
  te = (last >> 7) + 1u < static_cast<unsigned>(nt) ? static_cast<int>((last >> 7) + 1u) : nt;
  tb = 0;
  if (lo > pos0) {
    const unsigned dl = static_cast<unsigned>(lo - pos0) - 1u;
    const unsigned first = (step == 1 ? dl : dl / static_cast<unsigned>(step)) + 1u;  // first row with pos >= lo
    tb = first >= static_cast<unsigned>(len) ? nt : static_cast<int>(first >> 7);
  }
  if (tb > te) tb = te;
}

// ---------------------------------------------------------------- bf16 path
// Chunk tables that fit the plan itself (the common case: no extra memory, no
// copy). Larger problems, up to kTcMaxChunksAll chunks and kTcMaxKvSegsAll
// spans, keep the same tables in device memory (TcTables).
constexpr int kTcMaxChunks = 32;
constexpr int kTcMaxKvSegs = 64;
constexpr int kTcMaxChunksAll = 4096;
constexpr int kTcMaxKvSegsAll = 8192;
constexpr int kTcMaxQPiecesAll = 8192;  // query spans (the plan holds kMaxQPieces)
constexpr int kTcMaxOrder = 7936;  // q-tile pairs that can be LPT-ordered
constexpr int kTcRowsPerUnit = 256;  // two 128-row query tiles per work unit
constexpr int kTcMaxSkUnits = 320;   // units in the stream-K tail (< 2 x grid)
constexpr int kTcMaxGrid = 160;      // CTAs of one launch (one per SM)

// Scratch of the stream-K tail: one slot per CTA holds the partial results of
// the unit that CTA started mid-way (raw O, then per row m_ref, max, l, l_r),
// published by an epoch flag per query tile.
struct TcScratch {
  float* o;         // [grid][2][128][D]
  float4* stats;    // [grid][2][128]
  unsigned* flags;  // [grid][2]
};

struct alignas(128) TcPlan {
  CUtensorMap qmap;                  // Q  [B, Hq, Sq, D] bf16, box 64 x 128
  CUtensorMap omap;                  // O  [B, Hq, Sq, D] bf16, box 64 x 32 (when o_tma)
  CUtensorMap kmap[kTcMaxChunks];    // K chunk c [B, Hkv, len, D]
  CUtensorMap vmap[kTcMaxChunks];    // V chunk c
  void* out;                         // O (bf16) or u (fp32, stats mode)
  float* m;
  float* l;
  int64_t o_sb, o_sh, o_sr;          // element strides of out
  unsigned long long timeout_ns;     // budget of any single wait
  int32_t test_stall;                // test hook: MMA warp first waits on a barrier nobody arrives on
  int32_t B, Hq, Hkv, Sq;
  int32_t causal, stats_mode, ring, n_chunks;
  float scale, scale_log2;
  int32_t o_fp32;                    // ring mode: O written as fp32 instead of bf16
  int32_t o_tma;                     // bf16 O at head_dim 128 leaves through omap
  int32_t full_tiles;                // no causal mask, no documents, key spans of whole 128-row tiles
  int32_t mma_poll;                  // the MMA warp polls its barriers (two-pass form)
  int32_t n_qpieces, n_kvsegs, n_qpairs, has_order;
  int32_t n_units;
  // work split: every CTA first takes dp_rounds whole units round-robin, then
  // its share [sk_bound[c], sk_bound[c+1]) of the T key tiles of units
  // dp_rounds*G .. (laid end to end, sk_prefix[i] = first tile of unit i).
  // dp_snake: odd rounds hand the units to the CTAs in reverse order.
  // pair_block: the unit order's block of pair ranks (unit_coords).
  int32_t grid, dp_rounds, sk_units, sk_total, dp_snake, pair_block;
  unsigned epoch;                    // value a published partial carries
  TcScratch scratch;                 // null pointers when no unit is split
  int32_t sk_prefix[kTcMaxSkUnits + 1];
  int32_t sk_bound[kTcMaxGrid + 1];
  // first stream-K unit of CTA c: the last unit starting at or before
  // sk_bound[c], stepped back over empty units starting there (placed by the
  // host: the walk then starts with one read instead of a search)
  int16_t sk_first[kTcMaxGrid];
  int32_t chunk_seg_begin[kTcMaxChunks + 1];
  QPiece qp[kMaxQPieces];
  KvSeg ks[kTcMaxKvSegs];
  int32_t n_docs;                    // 0: no document mask
  int32_t doc_bounds[kMaxDocs + 1];
  // Device-resident chunk tables (null: the plan's own kmap, vmap, ks and
  // chunk_seg_begin hold them): tensor maps [n_chunks] each, spans
  // [n_kvsegs], first span of every chunk [n_chunks + 1].
  const CUtensorMap* ext_kmap;
  const CUtensorMap* ext_vmap;
  const KvSeg* ext_ks;
  const int32_t* ext_csb;
  const QPiece* ext_qp;              // query spans [n_qpieces] (null: qp)
  uint16_t order[kTcMaxOrder];       // q-pair visit order (longest first)
};
static_assert(sizeof(TcPlan) <= 32000, "bf16 plan must fit the parameter space");

// Byte layout of device-resident chunk tables (tensor maps first, 128-byte
// aligned): K maps, V maps, spans, first span per chunk.
struct TcTablesLayout {
  size_t kmap, vmap, ks, csb, qp, bytes;
  static TcTablesLayout of(int n_chunks, int n_segs, int n_qpieces) {
    TcTablesLayout t;
    t.kmap = 0;
    t.vmap = t.kmap + size_t(n_chunks) * sizeof(CUtensorMap);
    t.ks = t.vmap + size_t(n_chunks) * sizeof(CUtensorMap);
    t.csb = t.ks + size_t(n_segs) * sizeof(KvSeg);
    t.qp = (t.csb + size_t(n_chunks + 1) * sizeof(int32_t) + 15) & ~size_t(15);
    t.bytes = (t.qp + size_t(n_qpieces) * sizeof(QPiece) + 255) & ~size_t(255);
    return t;
  }
};

// ------------------------------------------------------- bf16 backward pass
// Gradients of the ring pass (dQ, and dK, dV of every chunk) in fp32. The
// row statistics of the forward are turned into lse2 = m log2(e) + log2(l)
// (so that P = exp2(s * scale * log2(e) - lse2)) and delta = sum_d dO * O by a
// preparation kernel; two tcgen05 kernels then recompute the probability
// tiles: one per key tile (dK, dV; every query row that sees the tile) and
// one per query tile (dQ; every key tile the rows see).
struct alignas(128) BwdPlan {
  CUtensorMap qmap;                  // Q  [B, Hq, Sq, D] bf16, box 64 x 128
  CUtensorMap domap;                 // dO [B, Hq, Sq, D] bf16
  CUtensorMap kmap[kTcMaxChunks];    // K chunk c [B, Hkv, len, D]
  CUtensorMap vmap[kTcMaxChunks];    // V chunk c
  const float* lse2;                 // [B, Hq, Sq]; +inf where the row sees no key
  const float* delta;                // [B, Hq, Sq]
  const int4* qtile_pos;             // [n_qtiles]: key windows of its rows: lowest lo,
                                     // highest hi, highest lo, lowest hi
  const uint8_t* colaux;             // [B * Hq][n_qtiles][kColAuxBytes]: per query tile
                                     // the dK/dV CTA's column data (see ra_bwd.cu)
  const uint16_t* q;                 // Q itself (bf16) and its element strides, read by the
  int64_t q_sb, q_sh, q_sr;          //   dQ CTAs into tensor memory
  float* dq;                         // [B, Hq, Sq, D] fp32, dense
  float* dk[kTcMaxChunks];           // [B, Hkv, len_c, D] fp32, dense
  float* dv[kTcMaxChunks];
  unsigned long long timeout_ns;
  int32_t B, Hq, Hkv, Sq;
  int32_t causal, n_chunks, n_qtiles, n_ktiles;
  float scale, scale_log2;
  int32_t n_qpieces, n_kvsegs;
  int32_t chunk_len[kTcMaxChunks];            // rows of chunk c (dk, dv row count)
  int32_t kseg_tile_begin[kTcMaxKvSegs + 1];  // first global key tile of span i
  QPiece qp[kMaxQPieces];
  KvSeg ks[kTcMaxKvSegs];
  int32_t n_docs;                             // 0: no document mask
  int32_t doc_bounds[kMaxDocs + 1];
  // Device-resident chunk tables (null: the plan's own arrays above), for
  // problems with more chunks or spans than the plan holds.
  const CUtensorMap* ext_kmap;                // [n_chunks]
  const CUtensorMap* ext_vmap;                // [n_chunks]
  float* const* ext_dk;                       // [n_chunks]
  float* const* ext_dv;                       // [n_chunks]
  const int32_t* ext_chunk_len;               // [n_chunks]
  const KvSeg* ext_ks;                        // [n_kvsegs]
  const int32_t* ext_ktb;                     // kseg_tile_begin [n_kvsegs + 1]
  const QPiece* ext_qp;                       // [n_qpieces]
};
static_assert(sizeof(BwdPlan) <= 32000, "backward plan must fit the parameter space");

// Column data of one 128-row query tile for the dK/dV CTAs, as it lies in
// shared memory: two K = 16 bias operand tiles (-lse2 / c and -delta, 4 KB
// each) and the rows' key windows (int2 lo, hi; 1 KB).
constexpr int kColAuxBytes = 2 * 4096 + 128 * 8;

// Byte layout of the backward's device-resident chunk tables.
struct BwdTablesLayout {
  size_t kmap, vmap, dk, dv, len, ks, ktb, qp, bytes;
  static BwdTablesLayout of(int n_chunks, int n_segs, int n_qpieces) {
    BwdTablesLayout t;
    t.kmap = 0;
    t.vmap = t.kmap + size_t(n_chunks) * sizeof(CUtensorMap);
    t.dk = t.vmap + size_t(n_chunks) * sizeof(CUtensorMap);
    t.dv = t.dk + size_t(n_chunks) * sizeof(float*);
    t.len = t.dv + size_t(n_chunks) * sizeof(float*);
    t.ks = (t.len + size_t(n_chunks) * sizeof(int32_t) + 15) & ~size_t(15);
    t.ktb = t.ks + size_t(n_segs) * sizeof(KvSeg);
    t.qp = (t.ktb + size_t(n_segs + 1) * sizeof(int32_t) + 15) & ~size_t(15);
    t.bytes = (t.qp + size_t(n_qpieces) * sizeof(QPiece) + 255) & ~size_t(255);
    return t;
  }
};

// ---------------------------------------------------------------- fp32 path
constexpr int kSimtMaxChunks = 256;
constexpr int kSimtMaxKvSegs = 320;

struct SimtChunk {
  const float* k;
  const float* v;
  int64_t k_sb, k_sh, k_sr, v_sb, v_sh, v_sr;
};

struct SimtPlan {
  const float* q;
  float* out;                        // O or u
  float* m;
  float* l;
  int64_t q_sb, q_sh, q_sr, o_sb, o_sh, o_sr;
  int32_t B, Hq, Hkv, D, Sq;
  int32_t causal, stats_mode, ring, n_chunks;
  int32_t n_qpieces, n_kvsegs;
  float scale;
  int32_t chunk_seg_begin[kSimtMaxChunks + 1];
  QPiece qp[kMaxQPieces];
  KvSeg ks[kSimtMaxKvSegs];
  SimtChunk ch[kSimtMaxChunks];
  int32_t n_docs;                    // 0: no document mask
  int32_t doc_bounds[kMaxDocs + 1];
};
static_assert(sizeof(SimtPlan) <= 32000, "fp32 plan must fit the parameter space");

// Bytes of stream-K scratch for a grid of `grid` CTAs: the raw O slots
// ([grid][2][128][D] fp32), the row statistics ([grid][2][128] float4) and the
// flags ([grid][2] u32), plus alignment slack.
constexpr size_t tc_scratch_bytes(int grid, int D) {
  return size_t(grid) * 2 * 128 * (size_t(D) * 4 + 16) + size_t(grid) * 2 * 4 + 256;
}

// Kernel launchers (defined in the .cu files; return a cudaError_t as int).
int launch_tc_bf16(const TcPlan& plan, int D, void* stream);
void tc_scratch_carve(void* base, int grid, int D, TcScratch* s);
// Device address of the fixed scratch array used by ra_ring_attention_noalloc
// on the current device (looked up once per device); returns a cudaError_t.
int tc_static_scratch(void** ptr, size_t* bytes);
int launch_simt_f32(const SimtPlan& plan, void* stream);
int launch_merge_f32(int64_t rows, int64_t D, float* u_acc, float* l_acc,
                     float* m_acc, const float* u_new, const float* l_new,
                     const float* m_new, int num_sms, void* stream);
int launch_merge_lse_f32(int64_t rows, int64_t D, float* o_acc, float* lse_acc, const float* o_new,
                         const float* lse_new, int num_sms, void* stream);
int launch_stats_to_lse(int64_t rows, const float* m, const float* l, float* lse, int num_sms,
                        void* stream);
int read_and_clear_device_error(int* code);
// Backward: the preparation kernels (lse2, delta, query-tile position ranges),
// then the dK/dV and dQ kernels; all on `stream`.
int launch_bwd_bf16(const BwdPlan& plan, int D, const void* o, int o_fp32, int64_t o_sb,
                    int64_t o_sh, int64_t o_sr, const void* dout, const float* m,
                    const float* l, float* lse2, float* delta, int4* qtile_pos, void* stream);
int read_and_clear_bwd_error(int* code);

}  // namespace ra
