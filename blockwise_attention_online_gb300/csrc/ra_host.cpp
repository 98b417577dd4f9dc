// Host side of the C ABI declared in include/ra.h: argument validation, plan
// building (position spans, ring visit order, causal work per query tile
// pair, longest-first order), TMA tensor-map creation and kernel launches.
//
// Plans travel as kernel parameters. Device memory is allocated only for the
// scratch of split units and for the device copies of the host-buffer entry
// point, stream-ordered, from one library pool per device.
#include "ra.h"

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <mutex>
#include <numeric>
#include <vector>

#include "ra_plan.h"

namespace {

thread_local char g_msg[512] = "";

ra_status fail(ra_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

ra_status ok() {
  g_msg[0] = '\0';
  return RA_OK;
}

constexpr int64_t kPosLimit = (int64_t(1) << 31) - 1;
// Weights of the stream-K split, in half key-tile steps: a plain step 2, the
// fixed cost of a unit 4 (measured: a unit switch costs about two steps of a
// long unit), 8 with packed documents (there a unit's fixed cost measured about
// four steps: 8 balanced 8K with documents of mean 1024 and 4096 best, +6% and
// +16% over 4), and a step of a unit whose rows lie in more than one packed
// document 3 (its rows have different key windows, so its steps mask element
// by element; of the factors tried, 1.5 balanced best).
constexpr int64_t kTileCost = 2;
constexpr int64_t kUnitCost = 4;
constexpr int64_t kUnitCostDocs = 8;
constexpr int64_t kMixedTileCost = 3;
constexpr int64_t kRowLimit = (int64_t(1) << 31) - 256;

// A flattened monotone span of rows with global positions.
struct Span {
  int64_t row0, len, pos0, step;
  int32_t owner;  // segment or chunk index
};

ra_status check_positions(const ra_positions& p, int64_t rows, const char* what,
                          int64_t idx) {
  if (p.nspan < 1 || p.nspan > RA_MAX_SPANS)
    return fail(RA_ERR_INVALID, "%s %lld: nspan=%d not in [1,%d]", what,
                (long long)idx, p.nspan, RA_MAX_SPANS);
  if (p.reserved != 0)
    return fail(RA_ERR_INVALID, "%s %lld: reserved field must be 0", what, (long long)idx);
  int64_t total = 0;
  for (int s = 0; s < p.nspan; ++s) {
    const ra_span& sp = p.span[s];
    if (sp.len < 0 || sp.pos0 < 0 || sp.step < 1)
      return fail(RA_ERR_INVALID, "%s %lld span %d: need len>=0, pos0>=0, step>=1",
                  what, (long long)idx, s);
    if (sp.len > 0) {
      // last position = pos0 + step*(len-1) must stay below 2^31-1
      if (sp.len - 1 > (kPosLimit - 1 - sp.pos0) / sp.step)
        return fail(RA_ERR_UNSUPPORTED, "%s %lld span %d: positions reach 2^31",
                    what, (long long)idx, s);
    }
    total += sp.len;
  }
  if (total != rows)
    return fail(RA_ERR_INVALID, "%s %lld: span lengths add to %lld, rows = %lld",
                what, (long long)idx, (long long)total, (long long)rows);
  return RA_OK;
}

struct Common {
  int64_t B, Hq, Hkv, D, Sq;
  int dtype, causal;
  float scale;
  int n_docs;                        // 0: no document mask
  std::vector<int32_t> doc_bounds;   // n_docs + 1 boundaries
  std::vector<Span> qspans;   // query pieces, owner = segment
  std::vector<Span> kvspans;  // key/value pieces, owner = chunk (row0 within chunk)
  std::vector<int> chunk_begin;  // kvspans of chunk c: [begin[c], begin[c+1])
  int nchunks;
  bool ring;
};

ra_status check_strides(const ra_strides& s, const char* what) {
  if (s.batch < 0 || s.head < 0 || s.row < 0)
    return fail(RA_ERR_INVALID, "%s: negative stride", what);
  return RA_OK;
}

// Document boundaries: strictly increasing, inside [0, 2^31 - 1], and every
// query and key position inside [b_0, b_n).
ra_status check_docs(const ra_problem& p, Common* c) {
  c->n_docs = 0;
  c->doc_bounds.clear();
  if (p.reserved_docs != 0) return fail(RA_ERR_INVALID, "reserved_docs must be 0");
  if (p.n_docs == 0) return RA_OK;
  if (p.n_docs < 0 || p.n_docs > RA_MAX_DOCS)
    return fail(RA_ERR_INVALID, "n_docs=%d not in [0,%d]", p.n_docs, RA_MAX_DOCS);
  if (!p.doc_bounds) return fail(RA_ERR_INVALID, "doc_bounds is NULL");
  for (int32_t d = 0; d <= p.n_docs; ++d) {
    const int64_t b = p.doc_bounds[d];
    if (b < 0 || b > kPosLimit)
      return fail(RA_ERR_INVALID, "doc_bounds[%d]=%lld outside [0, 2^31-1]", d, (long long)b);
    if (d > 0 && b <= p.doc_bounds[d - 1])
      return fail(RA_ERR_INVALID, "doc_bounds must increase strictly (index %d)", d);
    c->doc_bounds.push_back(int32_t(b));
  }
  const int64_t b0 = p.doc_bounds[0], bn = p.doc_bounds[p.n_docs];
  for (const std::vector<Span>* v : {&c->qspans, &c->kvspans})
    for (const Span& sp : *v)
      if (sp.pos0 < b0 || sp.pos0 + sp.step * (sp.len - 1) >= bn)
        return fail(RA_ERR_INVALID, "a position lies outside the documents [%lld, %lld)",
                    (long long)b0, (long long)bn);
  c->n_docs = p.n_docs;
  return RA_OK;
}

ra_status validate(const ra_problem* pb, const void* q, const ra_q_segment* segs,
                   int32_t nsegs, const ra_kv_chunk* chunks, int32_t nchunks,
                   Common* c) {
  if (!pb) return fail(RA_ERR_INVALID, "problem is NULL");
  const ra_problem& p = *pb;
  if (p.B < 1 || p.Hq < 1 || p.Hkv < 1 || p.D < 1 || p.Sq < 0)
    return fail(RA_ERR_INVALID, "need B, Hq, Hkv, D >= 1 and Sq >= 0");
  if (p.Hq % p.Hkv != 0)
    return fail(RA_ERR_INVALID, "Hq=%lld is not a multiple of Hkv=%lld",
                (long long)p.Hq, (long long)p.Hkv);
  if (p.dtype != RA_F32 && p.dtype != RA_BF16)
    return fail(RA_ERR_INVALID, "unknown dtype %d", p.dtype);
  if (p.causal != 0 && p.causal != 1) return fail(RA_ERR_INVALID, "causal must be 0 or 1");
  if (p.o_fp32 != 0 && p.o_fp32 != 1) return fail(RA_ERR_INVALID, "o_fp32 must be 0 or 1");
  if (!std::isfinite(p.scale)) return fail(RA_ERR_INVALID, "scale is not finite");
  if (p.dtype == RA_BF16 && p.D != 64 && p.D != 96 && p.D != 128)
    return fail(RA_ERR_UNSUPPORTED, "bf16 path supports head_dim 64, 96 or 128, got %lld",
                (long long)p.D);
  if (p.dtype == RA_F32 && p.D > 128)
    return fail(RA_ERR_UNSUPPORTED, "fp32 path supports head_dim <= 128, got %lld",
                (long long)p.D);
  if (p.Sq > kRowLimit) return fail(RA_ERR_UNSUPPORTED, "Sq too large");
  if (p.B * p.Hq > (int64_t(1) << 30)) return fail(RA_ERR_UNSUPPORTED, "B*Hq too large");
  ra_status st;
  if ((st = check_strides(p.q_strides, "q_strides")) != RA_OK) return st;
  if ((st = check_strides(p.o_strides, "o_strides")) != RA_OK) return st;
  if (p.Sq > 0 && !q) return fail(RA_ERR_INVALID, "q is NULL");
  if (nsegs < 0 || (nsegs > 0 && !segs)) return fail(RA_ERR_INVALID, "bad segment list");
  if (p.Sq > 0 && nsegs < 1) return fail(RA_ERR_INVALID, "need at least one query segment");
  if (nchunks < 0 || (nchunks > 0 && !chunks)) return fail(RA_ERR_INVALID, "bad chunk list");

  c->B = p.B; c->Hq = p.Hq; c->Hkv = p.Hkv; c->D = p.D; c->Sq = p.Sq;
  c->dtype = p.dtype; c->causal = p.causal;
  c->scale = p.scale > 0.f ? p.scale : float(1.0 / std::sqrt(double(p.D)));
  c->qspans.clear(); c->kvspans.clear(); c->chunk_begin.assign(1, 0);
  c->nchunks = nchunks;
  c->ring = (nsegs == nchunks && nchunks > 1);

  int64_t row = 0;
  for (int32_t s = 0; s < nsegs; ++s) {
    if (segs[s].len < 0) return fail(RA_ERR_INVALID, "segment %d: negative len", s);
    if ((st = check_positions(segs[s].pos, segs[s].len, "segment", s)) != RA_OK) return st;
    int64_t r = row;
    for (int k = 0; k < segs[s].pos.nspan; ++k) {
      const ra_span& sp = segs[s].pos.span[k];
      if (sp.len > 0) c->qspans.push_back({r, sp.len, sp.pos0, sp.len > 1 ? sp.step : 1, s});
      r += sp.len;
    }
    row += segs[s].len;
  }
  if (row != p.Sq)
    return fail(RA_ERR_INVALID, "segment lengths add to %lld, Sq = %lld",
                (long long)row, (long long)p.Sq);

  for (int32_t k = 0; k < nchunks; ++k) {
    const ra_kv_chunk& ch = chunks[k];
    if (ch.len < 0) return fail(RA_ERR_INVALID, "chunk %d: negative len", k);
    if (ch.len > kRowLimit) return fail(RA_ERR_UNSUPPORTED, "chunk %d too long", k);
    if ((st = check_positions(ch.pos, ch.len, "chunk", k)) != RA_OK) return st;
    if (ch.len > 0) {
      if (!ch.k || !ch.v) return fail(RA_ERR_INVALID, "chunk %d: NULL k or v", k);
      if ((st = check_strides(ch.k_strides, "chunk k_strides")) != RA_OK) return st;
      if ((st = check_strides(ch.v_strides, "chunk v_strides")) != RA_OK) return st;
      int64_t r = 0;
      for (int s = 0; s < ch.pos.nspan; ++s) {
        const ra_span& sp = ch.pos.span[s];
        if (sp.len > 0) c->kvspans.push_back({r, sp.len, sp.pos0, sp.len > 1 ? sp.step : 1, k});
        r += sp.len;
      }
    }
    c->chunk_begin.push_back(int(c->kvspans.size()));
  }
  if ((int64_t)c->qspans.size() > ra::kTcMaxQPiecesAll)
    return fail(RA_ERR_UNSUPPORTED, "%zu query spans exceed the limit of %d",
                c->qspans.size(), ra::kTcMaxQPiecesAll);
  return check_docs(p, c);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Lowest and highest position over query rows [r0, r1) (spans are sorted by
// row).
void qrange_of_rows(const std::vector<Span>& qs, int64_t r0, int64_t r1, int64_t* qmin,
                    int64_t* qmax) {
  *qmin = kPosLimit;
  *qmax = -1;
  for (const Span& s : qs) {
    int64_t a = std::max(r0, s.row0), b = std::min(r1, s.row0 + s.len);
    if (a < b) {
      *qmin = std::min(*qmin, s.pos0 + s.step * (a - s.row0));
      *qmax = std::max(*qmax, s.pos0 + s.step * (b - 1 - s.row0));
    }
  }
}

// Key tiles of a span (128 rows each) holding a position that some query in
// the position range [qmin, qmax] may see: the same count as the kernels'
// tile walk (both use ra::key_window and ra::live_range).
int64_t live_tiles(const Common& c, const Span& kv, int64_t qmin, int64_t qmax) {
  if (!c.causal && c.n_docs == 0) return (kv.len + 127) / 128;
  int lo, hi, unused;
  ra::key_window(c, int(qmin), lo, unused);
  ra::key_window(c, int(qmax), unused, hi);
  int tb, te;
  ra::live_range(int(kv.pos0), int(kv.step), int(kv.len), lo, hi, tb, te);
  return te - tb;
}

// ----------------------------------------------------------- tensor maps
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

ra_status get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return fail(RA_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  return RA_OK;
}

// 4-D bf16 map over [B, H, rows, D] with box 64 x box_rows (one 128-byte
// swizzle atom wide; a 128-row tile high unless given); rows past `rows`
// read as zero and are not written.
ra_status make_map(CUtensorMap* map, const void* base, int64_t D, int64_t rows,
                   int64_t H, int64_t B, const ra_strides& st, const char* what,
                   cuuint32_t box_rows = 128) {
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)rows, (cuuint64_t)H, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)st.row * 2, (cuuint64_t)st.head * 2,
                           (cuuint64_t)st.batch * 2};
  // unused axes (extent 1) may carry any stride; TMA still wants a multiple of 16
  if (rows == 1) strides[0] = std::max<cuuint64_t>(16, strides[0] & ~cuuint64_t(15));
  if (H == 1) strides[1] = std::max<cuuint64_t>(16, strides[1] & ~cuuint64_t(15));
  if (B == 1) strides[2] = std::max<cuuint64_t>(16, strides[2] & ~cuuint64_t(15));
  cuuint32_t box[4] = {64, box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base),
                        dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(RA_ERR_INVALID, "tensor map for %s rejected (CUresult %d)", what, (int)r);
  return RA_OK;
}

ra_status check_bf16_strides(const ra_strides& s, int64_t rows, int64_t H, int64_t B,
                             const char* what) {
  // TMA global strides must be multiples of 16 bytes (8 bf16 elements)
  if ((rows > 1 && s.row % 8) || (H > 1 && s.head % 8) || (B > 1 && s.batch % 8))
    return fail(RA_ERR_INVALID, "%s: bf16 strides must be multiples of 8 elements", what);
  if (rows > 1 && s.row < 1) return fail(RA_ERR_INVALID, "%s: zero row stride", what);
  return RA_OK;
}

int g_num_sms_cache[64];

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && g_num_sms_cache[dev] > 0) return g_num_sms_cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) g_num_sms_cache[dev] = n;
  return n;
}

ra_status cuda_status(int err, const char* what) {
  if (err == cudaSuccess) return ok();
  return fail(RA_ERR_CUDA, "%s: %s", what, cudaGetErrorString((cudaError_t)err));
}

// ----------------------------------------------------------- memory pool
// Stream-ordered allocations of the library come from one pool per device.
// The pool keeps up to kPoolKeepBytes mapped across synchronisations (the
// default pool would return everything at each synchronisation, and the next
// call would wait while memory is mapped again). It never makes a stream wait
// for another stream's free in order to reuse a block: calls on different
// streams stay independent, and the pool maps more memory instead.
constexpr uint64_t kPoolKeepBytes = uint64_t(4) << 30;

ra_status lib_pool(cudaMemPool_t* out) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static cudaMemPool_t pools[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_status(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(RA_ERR_UNSUPPORTED, "device %d out of range", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (!pools[dev]) {
    cudaMemPoolProps props;
    std::memset(&props, 0, sizeof(props));
    props.allocType = cudaMemAllocationTypePinned;
    props.handleTypes = cudaMemHandleTypeNone;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    e = cudaMemPoolCreate(&pool, &props);
    if (e != cudaSuccess) return cuda_status(e, "creating the library memory pool");
    uint64_t keep = kPoolKeepBytes;
    int no_cross_stream_wait = 0;
    e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
    if (e == cudaSuccess)
      e = cudaMemPoolSetAttribute(pool, cudaMemPoolReuseAllowInternalDependencies,
                                  &no_cross_stream_wait);
    if (e != cudaSuccess) {
      cudaMemPoolDestroy(pool);
      return cuda_status(e, "configuring the library memory pool");
    }
    pools[dev] = pool;
  }
  *out = pools[dev];
  return RA_OK;
}

// Enqueued on the launch stream after every check and plan has succeeded and
// right before the kernel launch (the host-buffer entry point copies its
// inputs here). Empty for the device-pointer entry points.
using BeforeLaunch = std::function<ra_status()>;

void fill_docs(const Common& c, int32_t* bounds, int32_t* n) {
  *n = c.n_docs;
  for (size_t i = 0; i < c.doc_bounds.size(); ++i) bounds[i] = c.doc_bounds[i];
}

// Query spans into `qp` (the plan's array when they fit, else `ext`, a
// byte buffer bound for device memory).
void fill_q_pieces(const Common& c, ra::QPiece* qp, int32_t* n, unsigned char* ext = nullptr) {
  *n = (int32_t)c.qspans.size();
  for (size_t i = 0; i < c.qspans.size(); ++i) {
    const Span& s = c.qspans[i];
    const ra::QPiece piece = {int32_t(s.row0), int32_t(s.len), int32_t(s.pos0), int32_t(s.step),
                              s.owner};
    if (ext)
      std::memcpy(ext + i * sizeof(ra::QPiece), &piece, sizeof(piece));
    else
      qp[i] = piece;
  }
}

// ----------------------------------------------------------- bf16 plan
// Where the scratch of a split launch comes from: a stream-ordered allocation
// for this call, or the library's fixed per-device array (no allocation).
enum class ScratchSource { kAllocate, kStatic };

ra_status run_tc(const Common& c, const ra_problem& p, const void* q,
                 const ra_kv_chunk* chunks, void* out, float* m, float* l,
                 bool stats_mode, void* stream, ScratchSource source,
                 const BeforeLaunch& before_launch) {
  if (c.nchunks > ra::kTcMaxChunksAll)
    return fail(RA_ERR_UNSUPPORTED, "bf16 path handles at most %d chunks, got %d",
                ra::kTcMaxChunksAll, c.nchunks);
  if ((int)c.kvspans.size() > ra::kTcMaxKvSegsAll)
    return fail(RA_ERR_UNSUPPORTED, "bf16 path handles at most %d chunk spans, got %zu",
                ra::kTcMaxKvSegsAll, c.kvspans.size());
  // chunk tables that do not fit the plan go to device memory
  const bool ext_tables = c.nchunks > ra::kTcMaxChunks ||
                          (int)c.kvspans.size() > ra::kTcMaxKvSegs ||
                          (int)c.qspans.size() > ra::kMaxQPieces;
  ra_status st;
  if (!aligned16(q)) return fail(RA_ERR_INVALID, "q must be 16-byte aligned");
  if (!aligned16(out)) return fail(RA_ERR_INVALID, "output must be 16-byte aligned");
  if ((st = check_bf16_strides(p.q_strides, c.Sq, c.Hq, c.B, "q_strides")) != RA_OK) return st;
  const bool out_f32 = stats_mode || p.o_fp32 == 1;
  const int64_t ovec = out_f32 ? 4 : 8;  // 16-byte row segments
  if ((c.Sq > 1 && p.o_strides.row % ovec) || (c.Hq > 1 && p.o_strides.head % ovec) ||
      (c.B > 1 && p.o_strides.batch % ovec))
    return fail(RA_ERR_INVALID, "output strides must be multiples of %lld elements",
                (long long)ovec);
  for (int k = 0; k < c.nchunks; ++k) {
    const ra_kv_chunk& ch = chunks[k];
    if (ch.len == 0) continue;
    if (!aligned16(ch.k) || !aligned16(ch.v))
      return fail(RA_ERR_INVALID, "chunk %d: k and v must be 16-byte aligned", k);
    if ((st = check_bf16_strides(ch.k_strides, ch.len, c.Hkv, c.B, "chunk k_strides")) != RA_OK) return st;
    if ((st = check_bf16_strides(ch.v_strides, ch.len, c.Hkv, c.B, "chunk v_strides")) != RA_OK) return st;
  }
  if ((st = get_encoder()) != RA_OK) return st;

  static thread_local ra::TcPlan plan;  // ~28 KB: keep it off the stack
  std::memset(&plan, 0, sizeof(plan));
  if ((st = make_map(&plan.qmap, q, c.D, std::max<int64_t>(c.Sq, 1), c.Hq, c.B,
                     p.q_strides, "q")) != RA_OK)
    return st;
  // bf16 O at head_dim 128: each softmax warp's 32 rows x 64 columns leave
  // its staging area in one asynchronous TMA store (box 64 x 32)
  if (!out_f32 && c.D == 128 && c.Sq > 0) {
    if ((st = make_map(&plan.omap, out, c.D, c.Sq, c.Hq, c.B, p.o_strides, "out", 32)) != RA_OK)
      return st;
    plan.o_tma = 1;
  }
  // device-resident tables are assembled here and copied in right before the
  // launch (the copy from pageable memory is staged, so this buffer may be
  // reused as soon as the copy call returns)
  static thread_local std::vector<unsigned char> tables;
  static thread_local std::vector<CUtensorMap> ext_maps;
  const ra::TcTablesLayout lay =
      ra::TcTablesLayout::of(ext_tables ? c.nchunks : 0, ext_tables ? int(c.kvspans.size()) : 0,
                             ext_tables ? int(c.qspans.size()) : 0);
  if (ext_tables) {
    ext_maps.assign(size_t(2) * c.nchunks, CUtensorMap{});
    tables.assign(lay.bytes, 0);
  }
  for (int k = 0; k < c.nchunks; ++k) {
    const ra_kv_chunk& ch = chunks[k];
    if (ch.len == 0) continue;
    CUtensorMap* km = ext_tables ? &ext_maps[k] : &plan.kmap[k];
    CUtensorMap* vm = ext_tables ? &ext_maps[c.nchunks + k] : &plan.vmap[k];
    if ((st = make_map(km, ch.k, c.D, ch.len, c.Hkv, c.B, ch.k_strides, "k")) != RA_OK) return st;
    if ((st = make_map(vm, ch.v, c.D, ch.len, c.Hkv, c.B, ch.v_strides, "v")) != RA_OK) return st;
  }
  plan.out = out; plan.m = m; plan.l = l;
  plan.o_sb = p.o_strides.batch; plan.o_sh = p.o_strides.head; plan.o_sr = p.o_strides.row;
  // Diagnostics: RA_WAIT_BUDGET_NS sets the budget of every on-chip wait
  // (default 2 s); RA_TEST_STALL=1 makes every CTA wait on a barrier that is
  // never completed, so that the bounded-wait path can be tested end to end.
  plan.timeout_ns = 2000000000ull;
  if (const char* e = std::getenv("RA_WAIT_BUDGET_NS")) {
    const long long v = std::atoll(e);
    if (v >= 1000) plan.timeout_ns = (unsigned long long)v;
  }
  if (const char* e = std::getenv("RA_TEST_STALL")) plan.test_stall = std::atoi(e) == 1;
  plan.B = int32_t(c.B); plan.Hq = int32_t(c.Hq); plan.Hkv = int32_t(c.Hkv);
  plan.Sq = int32_t(c.Sq);
  plan.causal = c.causal; plan.stats_mode = stats_mode ? 1 : 0;
  plan.ring = c.ring ? 1 : 0; plan.n_chunks = c.nchunks;
  plan.scale = c.scale;
  plan.scale_log2 = float(double(c.scale) * 1.4426950408889634);
  plan.o_fp32 = out_f32 ? 1 : 0;
  fill_q_pieces(c, plan.qp, &plan.n_qpieces, ext_tables ? tables.data() + lay.qp : nullptr);
  fill_docs(c, plan.doc_bounds, &plan.n_docs);
  plan.n_kvsegs = int32_t(c.kvspans.size());
  // every key tile whole and visible to every row: the softmax needs no
  // column bounds and no walk over the key spans
  plan.full_tiles = (!c.causal && plan.n_docs == 0) ? 1 : 0;
  for (const Span& kv : c.kvspans)
    if (kv.len % 128 != 0) plan.full_tiles = 0;
  if (ext_tables) {
    std::memcpy(tables.data() + lay.kmap, ext_maps.data(), size_t(2) * c.nchunks * sizeof(CUtensorMap));
    for (size_t i = 0; i < c.kvspans.size(); ++i) {
      const Span& s = c.kvspans[i];
      const ra::KvSeg kv = {s.owner, int32_t(s.row0), int32_t(s.len), int32_t(s.pos0),
                            int32_t(s.step), int32_t((s.len + 127) / 128)};
      std::memcpy(tables.data() + lay.ks + i * sizeof(ra::KvSeg), &kv, sizeof(kv));
    }
    std::memcpy(tables.data() + lay.csb, c.chunk_begin.data(), size_t(c.nchunks + 1) * sizeof(int32_t));
  } else {
    for (size_t i = 0; i < c.kvspans.size(); ++i) {
      const Span& s = c.kvspans[i];
      plan.ks[i] = {s.owner, int32_t(s.row0), int32_t(s.len), int32_t(s.pos0), int32_t(s.step),
                    int32_t((s.len + 127) / 128)};
    }
    for (int k = 0; k <= c.nchunks; ++k) plan.chunk_seg_begin[k] = c.chunk_begin[k];
  }

  const int64_t npairs = (c.Sq + ra::kTcRowsPerUnit - 1) / ra::kTcRowsPerUnit;
  plan.n_qpairs = int32_t(npairs);
  const int64_t BH = c.B * c.Hq;
  const int64_t units = npairs * BH;
  if (units > (int64_t(1) << 31) - 1) return fail(RA_ERR_UNSUPPORTED, "too many work units");
  plan.n_units = int32_t(units);
  if (units == 0) return ok();

  // live key tiles of every query-tile pair (the same for every head), and
  // the cost of one of its steps: a pair whose rows lie in more than one
  // packed document costs kMixedTileCost per step
  std::vector<int64_t> work(npairs, 0), step_cost(npairs, kTileCost);
  for (int64_t qp = 0; qp < npairs; ++qp) {
    int64_t r0 = qp * ra::kTcRowsPerUnit, r1 = std::min(c.Sq, r0 + ra::kTcRowsPerUnit);
    int64_t qmin, qmax;
    qrange_of_rows(c.qspans, r0, r1, &qmin, &qmax);
    for (const Span& kv : c.kvspans) work[qp] += live_tiles(c, kv, qmin, qmax);
    if (c.n_docs > 0) {
      int lo_min, lo_max, unused;
      ra::key_window(c, int(qmin), lo_min, unused);
      ra::key_window(c, int(qmax), lo_max, unused);
      if (lo_min != lo_max) step_cost[qp] = kMixedTileCost;  // different documents
    }
  }
  // visit order of the pairs: costliest first when the work differs
  // (causal, documents)
  std::vector<int32_t> order(npairs);
  std::iota(order.begin(), order.end(), 0);
  plan.has_order = 0;
  if (npairs <= ra::kTcMaxOrder && (c.causal || c.n_docs > 0)) {
    std::stable_sort(order.begin(), order.end(), [&](int32_t a, int32_t b) {
      return work[a] * step_cost[a] > work[b] * step_cost[b];
    });
    for (int64_t i = 0; i < npairs; ++i) plan.order[i] = uint16_t(order[i]);
    plan.has_order = 1;
  }
  int pair_block = 1;
  auto unit_rank = [&](int64_t u) {
    int rank, b, hq;
    ra::unit_coords(int(u), int(npairs), int(c.B), int(c.Hq), int(c.Hkv), pair_block, rank, b, hq);
    return rank;
  };
  auto unit_tiles = [&](int64_t u) { return work[order[unit_rank(u)]]; };
  auto unit_step_cost = [&](int64_t u) { return step_cost[order[unit_rank(u)]]; };

  const int sms = num_sms();
  if (sms <= 0) return cuda_status(cudaErrorNoDevice, "querying the SM count");
  int64_t total_tiles = 0;
  for (int64_t qp = 0; qp < npairs; ++qp) total_tiles += work[qp] * BH;
  // one CTA per SM; small problems use fewer CTAs (at least ~8 tiles each)
  int64_t G = std::min<int64_t>(std::min(sms, ra::kTcMaxGrid), std::max<int64_t>(1, total_tiles / 8));
  if (units >= G) G = std::min(sms, ra::kTcMaxGrid);
  // whole rounds stay data-parallel; the last one to two rounds are split by tiles
  int64_t R = units >= 2 * G ? units / G - 1 : 0;
  int64_t sk_units = units - R * G;
  if (sk_units > ra::kTcMaxSkUnits) {  // cannot happen with G <= kTcMaxGrid
    R = units / G;
    sk_units = units - R * G;
  }
  plan.grid = int32_t(G);
  plan.dp_rounds = int32_t(R);
  // Unit order of the whole-unit rounds. Pair-major units put every
  // key/value stream (batch, key/value head) into every round, so the units
  // sharing a stream's keys are few and far apart in time; with the long
  // causal launches most of the key/value stream then came from DRAM (128K
  // with 8 key/value heads: 171 GB per launch). Blocks of G / (Hq / Hkv)
  // pair ranks with the stream outermost make each round one stream's run of
  // consecutive pair ranks: 128K 7-11 GB and +4-5% on all three layouts, 1M
  // +10% (whose clock the power cap sets: less DRAM traffic, a higher
  // clock). A stream with fewer pair ranks than that would put several
  // streams' whole cost ranges into one round, which no CTA order balances
  // (16K causal with 16 heads: -13%), so such launches stay pair-major.
  // Inside a round the CTAs take the pair ranks in order, so alternate
  // rounds run in reverse CTA order; otherwise CTA 0 takes the costliest unit
  // of every round and the CTAs drift apart (32K causal: DRAM reads 21 GB
  // per launch with plain round-robin, 8.6 GB with the reversal).
  plan.dp_snake = R > 1 ? 1 : 0;
  const int64_t block = G / (c.Hq / c.Hkv);
  if (R > 1 && block >= 1 && npairs >= block) pair_block = int(block);
  plan.pair_block = pair_block;
  // The MMA warp polls its barriers unless the units are very long (more
  // than 1024 key tiles on average). Measured under the power cap: polling
  // raises the work per clock but lowers the clock the cap allows, and for
  // long units the second wins (512K causal: sleeping waits +0.8%, 1M +2%,
  // 1M with logits of +-60 +7%); up to 128K polling wins by 2-4%, sustained
  // runs included.
  plan.mma_poll = total_tiles <= int64_t(1024) * units ? 1 : 0;
  plan.sk_units = int32_t(sk_units);
  int64_t T = 0;
  plan.sk_prefix[0] = 0;
  for (int64_t i = 0; i < sk_units; ++i) {
    T += unit_tiles(R * G + i);
    plan.sk_prefix[i + 1] = int32_t(T);
  }
  if (T > (int64_t(1) << 30)) return fail(RA_ERR_UNSUPPORTED, "stream-K range too large");
  plan.sk_total = int32_t(T);
  // CTA boundaries on the tile line: each tail unit is weighed as its tiles
  // times its step cost plus unit_cost for the unit's fixed costs (its Q
  // load, the switch of the softmax warps, its epilogue), and the weighted
  // line is cut in G equal shares; a cut inside a unit's fixed cost moves to
  // its first tile. With equal units this is the plain cut of the tiles in G
  // shares; with many short units (causal starts, packed documents) or
  // costlier steps the CTAs that get them take fewer tiles.
  {
    const int64_t unit_cost = c.n_docs > 0 ? kUnitCostDocs : kUnitCost;
    int64_t W = 0;
    for (int64_t i = 0; i < sk_units; ++i)
      W += unit_cost + unit_step_cost(R * G + i) * (plan.sk_prefix[i + 1] - plan.sk_prefix[i]);
    int64_t i = 0, q = 0;  // unit i starts at weight q
    plan.sk_bound[0] = 0;
    for (int64_t c = 1; c <= G; ++c) {
      const int64_t x = c * W / G;
      while (i < sk_units) {
        const int64_t wi = unit_cost + unit_step_cost(R * G + i) *
                                           (plan.sk_prefix[i + 1] - plan.sk_prefix[i]);
        if (q + wi > x) break;
        q += wi;
        ++i;
      }
      const int64_t n = i < sk_units ? plan.sk_prefix[i + 1] - plan.sk_prefix[i] : 0;
      const int64_t f = i < sk_units ? unit_step_cost(R * G + i) : 1;
      const int64_t in = std::min(n, std::max<int64_t>(0, x - q - unit_cost) / f);
      plan.sk_bound[c] = int32_t(i < sk_units ? plan.sk_prefix[i] + in : T);
    }
    plan.sk_bound[G] = int32_t(T);
  }
  for (int64_t cta = 0; cta < G; ++cta) {
    const int64_t a = plan.sk_bound[cta];
    int64_t lo = 0, hi = sk_units - 1;
    while (lo < hi) {
      const int64_t mid = (lo + hi + 1) >> 1;
      if (plan.sk_prefix[mid] <= a) lo = mid; else hi = mid - 1;
    }
    while (lo > 0 && plan.sk_prefix[lo] == a && plan.sk_prefix[lo - 1] == a) --lo;
    plan.sk_first[cta] = int16_t(lo);
  }
  // does any CTA boundary fall strictly inside a unit?
  bool split = false;
  for (int64_t cta = 1; cta < G && !split; ++cta) {
    const int64_t a = plan.sk_bound[cta];
    for (int64_t i = 0; i < sk_units; ++i)
      if (plan.sk_prefix[i] < a && a < plan.sk_prefix[i + 1]) { split = true; break; }
  }
  static std::atomic<unsigned> epoch_counter{0};
  unsigned ep = ++epoch_counter;
  if (ep == 0) ep = ++epoch_counter;
  plan.epoch = ep;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const size_t scratch_bytes = split ? ra::tc_scratch_bytes(int(G), int(c.D)) : 0;
  const size_t tables_bytes = ext_tables ? lay.bytes : 0;
  // Device memory of this launch: the stream-K scratch at the start, the
  // chunk tables at the end; from the library pool (freed again after the
  // launch, stream-ordered) or from the fixed array (no allocation).
  char* mem = nullptr;
  size_t tables_off = 0;
  bool pooled = false;
  if (scratch_bytes + tables_bytes > 0) {
    if (source == ScratchSource::kStatic) {
      void* base = nullptr;
      size_t cap = 0;
      cudaError_t e = static_cast<cudaError_t>(ra::tc_static_scratch(&base, &cap));
      if (e != cudaSuccess) return cuda_status(e, "looking up the fixed scratch array");
      mem = static_cast<char*>(base);
      tables_off = (scratch_bytes + 255) & ~size_t(255);
      if (tables_off + tables_bytes > cap)
        return fail(RA_ERR_UNSUPPORTED,
                    "the launch needs %zu bytes of scratch and chunk tables, the fixed array holds %zu",
                    tables_off + tables_bytes, cap);
    } else {
      cudaMemPool_t pool = nullptr;
      if ((st = lib_pool(&pool)) != RA_OK) return st;
      tables_off = (scratch_bytes + 255) & ~size_t(255);
      cudaError_t e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&mem),
                                              tables_off + tables_bytes, pool, cs);
      if (e != cudaSuccess) return cuda_status(e, "allocating stream-K scratch and chunk tables");
      pooled = true;
    }
  }
  auto release = [&] {
    if (pooled) cudaFreeAsync(mem, cs);
  };
  if (split) ra::tc_scratch_carve(mem, int(G), int(c.D), &plan.scratch);
  if (ext_tables) {
    char* t = mem + tables_off;
    plan.ext_kmap = reinterpret_cast<const CUtensorMap*>(t + lay.kmap);
    plan.ext_vmap = reinterpret_cast<const CUtensorMap*>(t + lay.vmap);
    plan.ext_ks = reinterpret_cast<const ra::KvSeg*>(t + lay.ks);
    plan.ext_csb = reinterpret_cast<const int32_t*>(t + lay.csb);
    plan.ext_qp = reinterpret_cast<const ra::QPiece*>(t + lay.qp);
  }
  if (before_launch && (st = before_launch()) != RA_OK) {
    release();
    return st;
  }
  cudaError_t e = cudaSuccess;
  if (ext_tables)
    e = cudaMemcpyAsync(mem + tables_off, tables.data(), tables_bytes, cudaMemcpyHostToDevice, cs);
  // the flags of split units must start cleared (the fixed array keeps the
  // previous call's contents; a pool block may hold anything)
  if (e == cudaSuccess && split)
    e = cudaMemsetAsync(plan.scratch.flags, 0, size_t(G) * 2 * sizeof(unsigned), cs);
  if (e != cudaSuccess) {
    release();
    return cuda_status(e, "preparing the launch");
  }
  const int err = ra::launch_tc_bf16(plan, int(c.D), stream);
  release();
  return cuda_status(err, "bf16 ring kernel launch");
}

// ----------------------------------------------------------- fp32 plan
ra_status run_simt(const Common& c, const ra_problem& p, const void* q,
                   const ra_kv_chunk* chunks, void* out, float* m, float* l,
                   bool stats_mode, void* stream, const BeforeLaunch& before_launch) {
  if (c.nchunks > ra::kSimtMaxChunks)
    return fail(RA_ERR_UNSUPPORTED, "fp32 path handles at most %d chunks, got %d",
                ra::kSimtMaxChunks, c.nchunks);
  if ((int)c.kvspans.size() > ra::kSimtMaxKvSegs)
    return fail(RA_ERR_UNSUPPORTED, "fp32 path handles at most %d chunk spans, got %zu",
                ra::kSimtMaxKvSegs, c.kvspans.size());
  if ((int)c.qspans.size() > ra::kMaxQPieces)
    return fail(RA_ERR_UNSUPPORTED, "fp32 path handles at most %d query spans, got %zu",
                ra::kMaxQPieces, c.qspans.size());
  static thread_local ra::SimtPlan plan;
  std::memset(&plan, 0, sizeof(plan));
  plan.q = static_cast<const float*>(q);
  plan.out = static_cast<float*>(out); plan.m = m; plan.l = l;
  plan.q_sb = p.q_strides.batch; plan.q_sh = p.q_strides.head; plan.q_sr = p.q_strides.row;
  plan.o_sb = p.o_strides.batch; plan.o_sh = p.o_strides.head; plan.o_sr = p.o_strides.row;
  plan.B = int32_t(c.B); plan.Hq = int32_t(c.Hq); plan.Hkv = int32_t(c.Hkv);
  plan.D = int32_t(c.D); plan.Sq = int32_t(c.Sq);
  plan.causal = c.causal; plan.stats_mode = stats_mode ? 1 : 0;
  plan.ring = c.ring ? 1 : 0; plan.n_chunks = c.nchunks;
  plan.scale = c.scale;
  fill_q_pieces(c, plan.qp, &plan.n_qpieces);
  fill_docs(c, plan.doc_bounds, &plan.n_docs);
  plan.n_kvsegs = int32_t(c.kvspans.size());
  for (size_t i = 0; i < c.kvspans.size(); ++i) {
    const Span& s = c.kvspans[i];
    plan.ks[i] = {s.owner, int32_t(s.row0), int32_t(s.len), int32_t(s.pos0), int32_t(s.step),
                  int32_t((s.len + 31) / 32)};
  }
  for (int k = 0; k <= c.nchunks; ++k) plan.chunk_seg_begin[k] = c.chunk_begin[k];
  for (int k = 0; k < c.nchunks; ++k) {
    const ra_kv_chunk& ch = chunks[k];
    plan.ch[k] = {static_cast<const float*>(ch.k), static_cast<const float*>(ch.v),
                  ch.k_strides.batch, ch.k_strides.head, ch.k_strides.row,
                  ch.v_strides.batch, ch.v_strides.head, ch.v_strides.row};
  }
  if (c.Sq == 0) return ok();
  if (before_launch) {
    const ra_status hs = before_launch();
    if (hs != RA_OK) return hs;
  }
  return cuda_status(ra::launch_simt_f32(plan, stream), "fp32 ring kernel launch");
}

ra_status run(const ra_problem* pb, const void* q, const ra_q_segment* segs, int32_t nsegs,
              const ra_kv_chunk* chunks, int32_t nchunks, void* out, float* m, float* l,
              bool stats_mode, void* stream,
              ScratchSource source = ScratchSource::kAllocate,
              const BeforeLaunch& before_launch = BeforeLaunch()) {
  Common c;
  ra_status st = validate(pb, q, segs, nsegs, chunks, nchunks, &c);
  if (st != RA_OK) return st;
  if (c.Sq == 0) return ok();
  if (!out || !m || !l) return fail(RA_ERR_INVALID, "output pointer is NULL");
  if (c.dtype == RA_BF16)
    return run_tc(c, *pb, q, chunks, out, m, l, stats_mode, stream, source, before_launch);
  return run_simt(c, *pb, q, chunks, out, m, l, stats_mode, stream, before_launch);
}

// ----------------------------------------------------------- backward
ra_status run_bwd(const ra_problem* pb, const void* q, const ra_q_segment* segs, int32_t nsegs,
                  const ra_kv_chunk* chunks, int32_t nchunks, const void* o, const void* dout,
                  const float* m, const float* l, float* dq, const ra_kv_grad* grads,
                  void* stream) {
  Common c;
  ra_status st = validate(pb, q, segs, nsegs, chunks, nchunks, &c);
  if (st != RA_OK) return st;
  const ra_problem& p = *pb;
  if (c.dtype != RA_BF16)
    return fail(RA_ERR_UNSUPPORTED, "the backward pass is implemented for bf16 inputs only");
  if (c.D != 64 && c.D != 96 && c.D != 128)
    return fail(RA_ERR_UNSUPPORTED, "the backward pass supports head_dim 64, 96 or 128, got %lld",
                (long long)c.D);
  if (nchunks > 0 && !grads) return fail(RA_ERR_INVALID, "grads is NULL");
  for (int32_t k = 0; k < nchunks; ++k)
    if (chunks[k].len > 0 && (!grads[k].dk || !grads[k].dv))
      return fail(RA_ERR_INVALID, "chunk %d: NULL dk or dv", k);
  if (c.nchunks > ra::kTcMaxChunksAll)
    return fail(RA_ERR_UNSUPPORTED, "bf16 path handles at most %d chunks, got %d",
                ra::kTcMaxChunksAll, c.nchunks);
  if ((int)c.kvspans.size() > ra::kTcMaxKvSegsAll)
    return fail(RA_ERR_UNSUPPORTED, "bf16 path handles at most %d chunk spans, got %zu",
                ra::kTcMaxKvSegsAll, c.kvspans.size());
  const bool ext_tables = c.nchunks > ra::kTcMaxChunks ||
                          (int)c.kvspans.size() > ra::kTcMaxKvSegs ||
                          (int)c.qspans.size() > ra::kMaxQPieces;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (c.Sq > 0) {
    if (!o || !dout || !m || !l || !dq) return fail(RA_ERR_INVALID, "o, dout, m, l or dq is NULL");
    if (!aligned16(q) || !aligned16(o) || !aligned16(dout) || !aligned16(dq))
      return fail(RA_ERR_INVALID, "q, o, dout and dq must be 16-byte aligned");
    if ((st = check_bf16_strides(p.q_strides, c.Sq, c.Hq, c.B, "q_strides")) != RA_OK) return st;
    // dO (bf16) shares O's element strides; they must suit both
    if ((st = check_bf16_strides(p.o_strides, c.Sq, c.Hq, c.B, "o_strides (dout)")) != RA_OK)
      return st;
  }
  for (int k = 0; k < c.nchunks; ++k) {
    const ra_kv_chunk& ch = chunks[k];
    if (ch.len == 0) continue;
    if (!aligned16(ch.k) || !aligned16(ch.v) || !aligned16(grads[k].dk) || !aligned16(grads[k].dv))
      return fail(RA_ERR_INVALID, "chunk %d: k, v, dk and dv must be 16-byte aligned", k);
    if ((st = check_bf16_strides(ch.k_strides, ch.len, c.Hkv, c.B, "chunk k_strides")) != RA_OK) return st;
    if ((st = check_bf16_strides(ch.v_strides, ch.len, c.Hkv, c.B, "chunk v_strides")) != RA_OK) return st;
  }
  if (c.Sq == 0) {
    // no query: every key and value gradient is zero
    for (int k = 0; k < c.nchunks; ++k) {
      if (chunks[k].len == 0) continue;
      const size_t bytes = size_t(c.B * c.Hkv * chunks[k].len) * size_t(c.D) * 4;
      cudaError_t e = cudaMemsetAsync(grads[k].dk, 0, bytes, cs);
      if (e == cudaSuccess) e = cudaMemsetAsync(grads[k].dv, 0, bytes, cs);
      if (e != cudaSuccess) return cuda_status(e, "clearing dk, dv");
    }
    return ok();
  }
  if ((st = get_encoder()) != RA_OK) return st;

  static thread_local ra::BwdPlan plan;
  std::memset(&plan, 0, sizeof(plan));
  if ((st = make_map(&plan.qmap, q, c.D, c.Sq, c.Hq, c.B, p.q_strides, "q")) != RA_OK) return st;
  plan.q = static_cast<const uint16_t*>(q);
  plan.q_sb = p.q_strides.batch; plan.q_sh = p.q_strides.head; plan.q_sr = p.q_strides.row;
  if ((st = make_map(&plan.domap, dout, c.D, c.Sq, c.Hq, c.B, p.o_strides, "dout")) != RA_OK)
    return st;
  // chunk tables: in the plan, or assembled here for device memory
  const ra::BwdTablesLayout lay = ra::BwdTablesLayout::of(
      ext_tables ? c.nchunks : 0, ext_tables ? int(c.kvspans.size()) : 0,
      ext_tables ? int(c.qspans.size()) : 0);
  static thread_local std::vector<CUtensorMap> ext_maps;
  static thread_local std::vector<unsigned char> tables;
  if (ext_tables) {
    ext_maps.assign(size_t(2) * c.nchunks, CUtensorMap{});
    tables.assign(lay.bytes, 0);
  }
  for (int k = 0; k < c.nchunks; ++k) {
    const ra_kv_chunk& ch = chunks[k];
    const int32_t len = int32_t(ch.len);
    float* dkp = ch.len ? grads[k].dk : nullptr;
    float* dvp = ch.len ? grads[k].dv : nullptr;
    if (ext_tables) {
      std::memcpy(tables.data() + lay.len + k * sizeof(int32_t), &len, sizeof(len));
      std::memcpy(tables.data() + lay.dk + k * sizeof(float*), &dkp, sizeof(dkp));
      std::memcpy(tables.data() + lay.dv + k * sizeof(float*), &dvp, sizeof(dvp));
    } else {
      plan.chunk_len[k] = len;
      plan.dk[k] = dkp;
      plan.dv[k] = dvp;
    }
    if (ch.len == 0) continue;
    CUtensorMap* km = ext_tables ? &ext_maps[k] : &plan.kmap[k];
    CUtensorMap* vm = ext_tables ? &ext_maps[c.nchunks + k] : &plan.vmap[k];
    if ((st = make_map(km, ch.k, c.D, ch.len, c.Hkv, c.B, ch.k_strides, "k")) != RA_OK) return st;
    if ((st = make_map(vm, ch.v, c.D, ch.len, c.Hkv, c.B, ch.v_strides, "v")) != RA_OK) return st;
  }
  plan.dq = dq;
  plan.timeout_ns = 2000000000ull;
  if (const char* env = std::getenv("RA_WAIT_BUDGET_NS")) {
    const unsigned long long v = std::strtoull(env, nullptr, 10);
    if (v > 0) plan.timeout_ns = v;
  }
  plan.B = int32_t(c.B); plan.Hq = int32_t(c.Hq); plan.Hkv = int32_t(c.Hkv); plan.Sq = int32_t(c.Sq);
  plan.causal = c.causal; plan.n_chunks = c.nchunks;
  plan.scale = c.scale;
  plan.scale_log2 = float(double(c.scale) * 1.4426950408889634);
  fill_q_pieces(c, plan.qp, &plan.n_qpieces, ext_tables ? tables.data() + lay.qp : nullptr);
  fill_docs(c, plan.doc_bounds, &plan.n_docs);
  plan.n_kvsegs = int32_t(c.kvspans.size());
  int64_t tiles = 0;
  for (size_t i = 0; i < c.kvspans.size(); ++i) {
    const Span& sp = c.kvspans[i];
    const ra::KvSeg kv = {sp.owner, int32_t(sp.row0), int32_t(sp.len), int32_t(sp.pos0),
                          int32_t(sp.step), int32_t((sp.len + 127) / 128)};
    const int32_t t0 = int32_t(tiles);
    if (ext_tables) {
      std::memcpy(tables.data() + lay.ks + i * sizeof(ra::KvSeg), &kv, sizeof(kv));
      std::memcpy(tables.data() + lay.ktb + i * sizeof(int32_t), &t0, sizeof(t0));
    } else {
      plan.ks[i] = kv;
      plan.kseg_tile_begin[i] = t0;
    }
    tiles += kv.ntiles;
  }
  if (tiles > (int64_t(1) << 30)) return fail(RA_ERR_UNSUPPORTED, "too many key tiles");
  {
    const int32_t tn = int32_t(tiles);
    if (ext_tables)
      std::memcpy(tables.data() + lay.ktb + c.kvspans.size() * sizeof(int32_t), &tn, sizeof(tn));
    else
      plan.kseg_tile_begin[c.kvspans.size()] = tn;
  }
  if (ext_tables)
    std::memcpy(tables.data() + lay.kmap, ext_maps.data(), size_t(2) * c.nchunks * sizeof(CUtensorMap));
  plan.n_ktiles = int32_t(tiles);
  plan.n_qtiles = int32_t((c.Sq + 127) / 128);
  if (int64_t(plan.n_ktiles) * c.Hkv * c.B > (int64_t(1) << 31) - 1 ||
      int64_t(plan.n_qtiles) * c.Hq * c.B > (int64_t(1) << 31) - 1)
    return fail(RA_ERR_UNSUPPORTED, "too many tiles for one launch");

  // per query row: lse2, delta; per query tile: key window bounds
  const size_t rows = size_t(c.B * c.Hq * c.Sq);
  auto up = [](size_t n) { return (n + 255) & ~size_t(255); };
  const size_t colaux_off = 2 * up(rows * 4) + up(size_t(plan.n_qtiles) * 16);
  const size_t colaux_bytes = size_t(c.B * c.Hq) * size_t(plan.n_qtiles) * ra::kColAuxBytes;
  const size_t tables_off = colaux_off + up(colaux_bytes);
  const size_t bytes = tables_off + (ext_tables ? lay.bytes : 0);
  cudaMemPool_t pool = nullptr;
  if ((st = lib_pool(&pool)) != RA_OK) return st;
  char* scratch = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&scratch), bytes, pool, cs);
  if (e != cudaSuccess) return cuda_status(e, "allocating backward scratch");
  float* lse2 = reinterpret_cast<float*>(scratch);
  float* delta = reinterpret_cast<float*>(scratch + up(rows * 4));
  int4* qtile_pos = reinterpret_cast<int4*>(scratch + 2 * up(rows * 4));
  plan.lse2 = lse2;
  plan.delta = delta;
  plan.qtile_pos = qtile_pos;
  plan.colaux = reinterpret_cast<const uint8_t*>(scratch + colaux_off);
  if (ext_tables) {
    char* t = scratch + tables_off;
    plan.ext_kmap = reinterpret_cast<const CUtensorMap*>(t + lay.kmap);
    plan.ext_vmap = reinterpret_cast<const CUtensorMap*>(t + lay.vmap);
    plan.ext_dk = reinterpret_cast<float* const*>(t + lay.dk);
    plan.ext_dv = reinterpret_cast<float* const*>(t + lay.dv);
    plan.ext_chunk_len = reinterpret_cast<const int32_t*>(t + lay.len);
    plan.ext_ks = reinterpret_cast<const ra::KvSeg*>(t + lay.ks);
    plan.ext_ktb = reinterpret_cast<const int32_t*>(t + lay.ktb);
    plan.ext_qp = reinterpret_cast<const ra::QPiece*>(t + lay.qp);
    // staged copy from pageable memory: the buffer may be reused once it returns
    e = cudaMemcpyAsync(t, tables.data(), lay.bytes, cudaMemcpyHostToDevice, cs);
    if (e != cudaSuccess) {
      cudaFreeAsync(scratch, cs);
      return cuda_status(e, "copying the chunk tables");
    }
  }
  const bool o_f32 = p.o_fp32 == 1;
  const int err = ra::launch_bwd_bf16(plan, int(c.D), o, o_f32 ? 1 : 0, p.o_strides.batch,
                                      p.o_strides.head, p.o_strides.row, dout, m, l, lse2, delta,
                                      qtile_pos, stream);
  cudaFreeAsync(scratch, cs);
  return cuda_status(err, "backward kernel launch");
}

// Dense strides of a [B, H, rows, D] tensor; axes of extent 1 accept any stride.
bool is_dense(const ra_strides& s, int64_t B, int64_t H, int64_t rows, int64_t D) {
  return (rows <= 1 || s.row == D) && (H <= 1 || s.head == rows * D) &&
         (B <= 1 || s.batch == H * rows * D);
}

// Start of the allocation that holds host pointer p (pinned memory the driver
// knows), or 0 when the driver cannot tell.
uintptr_t host_allocation_start(const void* p) {
  static PFN_cuPointerGetAttribute_v4000 get_attr = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuPointerGetAttribute", &fn, 4000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_attr = reinterpret_cast<PFN_cuPointerGetAttribute_v4000>(fn);
  });
  CUdeviceptr start = 0;
  if (!get_attr || !p ||
      get_attr(&start, CU_POINTER_ATTRIBUTE_RANGE_START_ADDR, reinterpret_cast<CUdeviceptr>(p)) !=
          CUDA_SUCCESS)
    return 0;
  return static_cast<uintptr_t>(start);
}

// One host<->device copy. A copy whose source and destination both continue
// the previous one's is merged into it, but only inside one host allocation
// (`host_alloc`, 0 if unknown: never merged); the device side is always one
// pool allocation.
struct Copy {
  char* dst;
  const char* src;
  size_t n;
  uintptr_t host_alloc;
};

void add_copy(std::vector<Copy>& v, void* dst, const void* src, size_t n, uintptr_t host_alloc) {
  if (n == 0) return;
  char* d = static_cast<char*>(dst);
  const char* s = static_cast<const char*>(src);
  if (!v.empty() && host_alloc != 0 && v.back().host_alloc == host_alloc &&
      v.back().dst + v.back().n == d && v.back().src + v.back().n == s) {
    v.back().n += n;
    return;
  }
  v.push_back({d, s, n, host_alloc});
}

cudaError_t issue_copies(const std::vector<Copy>& v, cudaMemcpyKind kind, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  for (size_t i = 0; e == cudaSuccess && i < v.size(); ++i)
    e = cudaMemcpyAsync(v[i].dst, v[i].src, v[i].n, kind, s);
  return e;
}

ra_status run_host(const ra_problem* pb, const void* q, const ra_q_segment* segs, int32_t nsegs,
                   const ra_kv_chunk* chunks, int32_t nchunks, void* o, float* m, float* l,
                   void* stream) {
  Common c;
  ra_status st = validate(pb, q, segs, nsegs, chunks, nchunks, &c);
  if (st != RA_OK) return st;
  if (c.Sq == 0) return ok();
  if (!o || !m || !l) return fail(RA_ERR_INVALID, "output pointer is NULL");
  const ra_problem& p = *pb;
  if (!is_dense(p.q_strides, c.B, c.Hq, c.Sq, c.D)) return fail(RA_ERR_INVALID, "host q must be dense");
  if (!is_dense(p.o_strides, c.B, c.Hq, c.Sq, c.D)) return fail(RA_ERR_INVALID, "host o must be dense");
  for (int32_t k = 0; k < nchunks; ++k) {
    const ra_kv_chunk& ch = chunks[k];
    if (ch.len > 0 && (!is_dense(ch.k_strides, c.B, c.Hkv, ch.len, c.D) ||
                       !is_dense(ch.v_strides, c.B, c.Hkv, ch.len, c.D)))
      return fail(RA_ERR_INVALID, "host chunk %d: k and v must be dense", k);
  }
  const size_t es = p.dtype == RA_BF16 ? 2 : 4;
  const size_t oes = (p.dtype == RA_BF16 && p.o_fp32 == 1) ? 4 : es;
  auto up = [](size_t n) { return (n + 255) & ~size_t(255); };
  const size_t rows = size_t(c.B * c.Hq * c.Sq);
  const size_t q_bytes = rows * size_t(c.D) * es, o_bytes = rows * size_t(c.D) * oes;
  size_t total = up(q_bytes) + up(o_bytes) + 2 * up(rows * 4);
  std::vector<size_t> kv_bytes(nchunks, 0);
  for (int32_t k = 0; k < nchunks; ++k) {
    kv_bytes[k] = size_t(c.B * c.Hkv * chunks[k].len) * size_t(c.D) * es;
    total += 2 * up(kv_bytes[k]);
  }
  cudaMemPool_t pool = nullptr;
  if ((st = lib_pool(&pool)) != RA_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  char* base = nullptr;
  cudaError_t e = cudaMallocFromPoolAsync(reinterpret_cast<void**>(&base), total, pool, cs);
  if (e != cudaSuccess) return cuda_status(e, "allocating device copies");
  // carve: o, m, l, then q, the k of every chunk and the v of every chunk, in
  // that order, so that inputs adjacent on the host are adjacent here too
  char* at = base;
  auto take = [&](size_t n) { char* r = at; at += up(n); return r; };
  void* dout = take(o_bytes);
  float* dm = reinterpret_cast<float*>(take(rows * 4));
  float* dl = reinterpret_cast<float*>(take(rows * 4));
  void* dq = take(q_bytes);
  std::vector<ra_kv_chunk> dch(chunks, chunks + nchunks);
  std::vector<void*> dk(nchunks, nullptr), dv(nchunks, nullptr);
  for (int32_t k = 0; k < nchunks; ++k)
    if (chunks[k].len > 0) dk[k] = take(kv_bytes[k]);
  for (int32_t k = 0; k < nchunks; ++k)
    if (chunks[k].len > 0) dv[k] = take(kv_bytes[k]);
  for (int32_t k = 0; k < nchunks; ++k) {
    dch[k].k = dk[k];
    dch[k].v = dv[k];
  }
  // the copies, with runs that are adjacent both on the host and on the device
  // merged into one (q, then the k and v of chunk-major buffers; o, m, l)
  std::vector<Copy> in, out;
  auto h2d = [&](void* dst, const void* src, size_t n) {
    add_copy(in, dst, src, n, n ? host_allocation_start(src) : 0);
  };
  auto d2h = [&](void* dst, const void* src, size_t n) {
    add_copy(out, dst, src, n, n ? host_allocation_start(dst) : 0);
  };
  h2d(dq, q, q_bytes);
  for (int32_t k = 0; k < nchunks; ++k) h2d(dk[k], chunks[k].k, kv_bytes[k]);
  for (int32_t k = 0; k < nchunks; ++k) h2d(dv[k], chunks[k].v, kv_bytes[k]);
  d2h(o, dout, o_bytes);
  d2h(m, dm, rows * 4);
  d2h(l, dl, rows * 4);
  ra_problem dp = p;
  const ra_strides dense_q = {c.Hq * c.Sq * c.D, c.Sq * c.D, c.D};
  dp.q_strides = dense_q;
  dp.o_strides = dense_q;
  for (int32_t k = 0; k < nchunks; ++k) {
    const ra_strides ds = {c.Hkv * chunks[k].len * c.D, chunks[k].len * c.D, c.D};
    dch[k].k_strides = ds;
    dch[k].v_strides = ds;
  }
  // issued only once the plan has been accepted
  const BeforeLaunch copy_in = [&]() -> ra_status {
    return cuda_status(issue_copies(in, cudaMemcpyHostToDevice, cs),
                       "copying inputs to the device");
  };
  st = run(&dp, dq, segs, nsegs, dch.data(), nchunks, dout, dm, dl, false, stream,
           ScratchSource::kAllocate, copy_in);
  if (st == RA_OK)
    st = cuda_status(issue_copies(out, cudaMemcpyDeviceToHost, cs), "copying outputs to the host");
  cudaFreeAsync(base, cs);
  return st;
}

}  // namespace

extern "C" {

ra_status ra_chunk_stats(const ra_problem* problem, const void* q,
                         const ra_q_segment* segs, int32_t nsegs,
                         const ra_kv_chunk* chunk, float* u, float* l, float* m,
                         void* stream) {
  if (!chunk) return fail(RA_ERR_INVALID, "chunk is NULL");
  return run(problem, q, segs, nsegs, chunk, 1, u, m, l, true, stream);
}

ra_status ra_ring_attention(const ra_problem* problem, const void* q,
                            const ra_q_segment* segs, int32_t nsegs,
                            const ra_kv_chunk* chunks, int32_t nchunks, void* o,
                            float* m, float* l, void* stream) {
  return run(problem, q, segs, nsegs, chunks, nchunks, o, m, l, false, stream);
}

ra_status ra_ring_attention_noalloc(const ra_problem* problem, const void* q,
                                    const ra_q_segment* segs, int32_t nsegs,
                                    const ra_kv_chunk* chunks, int32_t nchunks, void* o,
                                    float* m, float* l, void* stream) {
  return run(problem, q, segs, nsegs, chunks, nchunks, o, m, l, false, stream,
             ScratchSource::kStatic);
}

ra_status ra_ring_attention_bwd(const ra_problem* problem, const void* q,
                                const ra_q_segment* segs, int32_t nsegs,
                                const ra_kv_chunk* chunks, int32_t nchunks, const void* o,
                                const void* dout, const float* m, const float* l, float* dq,
                                const ra_kv_grad* grads, void* stream) {
  return run_bwd(problem, q, segs, nsegs, chunks, nchunks, o, dout, m, l, dq, grads, stream);
}

ra_status ra_ring_attention_host(const ra_problem* problem, const void* q,
                                 const ra_q_segment* segs, int32_t nsegs,
                                 const ra_kv_chunk* chunks, int32_t nchunks, void* o,
                                 float* m, float* l, void* stream) {
  return run_host(problem, q, segs, nsegs, chunks, nchunks, o, m, l, stream);
}

ra_status ra_merge_stats(int64_t rows, int64_t D, float* u_acc, float* l_acc, float* m_acc,
                         const float* u_new, const float* l_new, const float* m_new,
                         void* stream) {
  if (rows < 0 || D < 1) return fail(RA_ERR_INVALID, "need rows >= 0 and D >= 1");
  if (rows == 0) return ok();
  if (!u_acc || !l_acc || !m_acc || !u_new || !l_new || !m_new)
    return fail(RA_ERR_INVALID, "NULL pointer");
  if (rows > (int64_t(1) << 40) / D) return fail(RA_ERR_UNSUPPORTED, "too many elements");
  const int sms = num_sms();
  if (sms <= 0) return cuda_status(cudaErrorNoDevice, "querying the SM count");
  return cuda_status(ra::launch_merge_f32(rows, D, u_acc, l_acc, m_acc, u_new, l_new, m_new,
                                          sms, stream),
                     "merge kernel launch");
}

ra_status ra_merge_lse(int64_t rows, int64_t D, float* o_acc, float* lse_acc, const float* o_new,
                       const float* lse_new, void* stream) {
  if (rows < 0 || D < 1) return fail(RA_ERR_INVALID, "need rows >= 0 and D >= 1");
  if (rows == 0) return ok();
  if (!o_acc || !lse_acc || !o_new || !lse_new) return fail(RA_ERR_INVALID, "NULL pointer");
  if (rows > (int64_t(1) << 40) / D) return fail(RA_ERR_UNSUPPORTED, "too many elements");
  const int sms = num_sms();
  if (sms <= 0) return cuda_status(cudaErrorNoDevice, "querying the SM count");
  return cuda_status(ra::launch_merge_lse_f32(rows, D, o_acc, lse_acc, o_new, lse_new, sms, stream),
                     "lse merge kernel launch");
}

ra_status ra_stats_to_lse(int64_t rows, const float* m, const float* l, float* lse, void* stream) {
  if (rows < 0) return fail(RA_ERR_INVALID, "need rows >= 0");
  if (rows == 0) return ok();
  if (!m || !l || !lse) return fail(RA_ERR_INVALID, "NULL pointer");
  const int sms = num_sms();
  if (sms <= 0) return cuda_status(cudaErrorNoDevice, "querying the SM count");
  return cuda_status(ra::launch_stats_to_lse(rows, m, l, lse, sms, stream), "lse kernel launch");
}

ra_status ra_segment_work(const ra_problem* problem, const ra_q_segment* segs, int32_t nsegs,
                          const ra_kv_chunk* chunks, int32_t nchunks, int64_t* pairs,
                          int64_t* tiles) {
  Common c;
  // positions only: pointers are not needed for bookkeeping
  ra_status st = validate(problem, reinterpret_cast<const void*>(16), segs, nsegs, nullptr,
                          0, &c);
  if (st != RA_OK) return st;
  if (nchunks < 0 || (nchunks > 0 && !chunks)) return fail(RA_ERR_INVALID, "bad chunk list");
  std::vector<Span> kv;
  for (int32_t k = 0; k < nchunks; ++k) {
    if (chunks[k].len < 0) return fail(RA_ERR_INVALID, "chunk %d: negative len", k);
    if ((st = check_positions(chunks[k].pos, chunks[k].len, "chunk", k)) != RA_OK) return st;
    int64_t r = 0;
    for (int s = 0; s < chunks[k].pos.nspan; ++s) {
      const ra_span& sp = chunks[k].pos.span[s];
      if (sp.len > 0) kv.push_back({r, sp.len, sp.pos0, sp.len > 1 ? sp.step : 1, k});
      r += sp.len;
    }
  }
  if (c.n_docs > 0) {
    // the same rule as the launches: every key position inside [b_0, b_n)
    const int64_t b0 = c.doc_bounds.front(), bn = c.doc_bounds.back();
    for (const Span& sp : kv)
      if (sp.pos0 < b0 || sp.pos0 + sp.step * (sp.len - 1) >= bn)
        return fail(RA_ERR_INVALID, "a position lies outside the documents [%lld, %lld)",
                    (long long)b0, (long long)bn);
  }
  for (int32_t s = 0; s < nsegs; ++s) {
    if (pairs) pairs[s] = 0;
    if (tiles) tiles[s] = 0;
  }
  if (pairs) {
    for (const Span& qs : c.qspans) {
      int64_t acc = 0;
      for (int64_t i = 0; i < qs.len; ++i) {
        int64_t pq = qs.pos0 + qs.step * i;
        if (!c.causal && c.n_docs == 0) {
          for (const Span& ks : kv) acc += ks.len;
          continue;
        }
        int lo, hi;
        ra::key_window(c, int(pq), lo, hi);
        for (const Span& ks : kv) {
          // rows with lo <= pos0 + step * r <= hi
          if (hi < ks.pos0) continue;
          const int64_t r_hi = std::min(ks.len - 1, (hi - ks.pos0) / ks.step);
          const int64_t r_lo = lo <= ks.pos0 ? 0 : (lo - ks.pos0 - 1) / ks.step + 1;
          if (r_hi >= r_lo) acc += r_hi - r_lo + 1;
        }
      }
      pairs[qs.owner] += acc;
    }
  }
  if (tiles) {
    const int64_t npairs = (c.Sq + ra::kTcRowsPerUnit - 1) / ra::kTcRowsPerUnit;
    for (int64_t qp = 0; qp < npairs; ++qp) {
      int64_t r0 = qp * ra::kTcRowsPerUnit, r1 = std::min(c.Sq, r0 + ra::kTcRowsPerUnit);
      int64_t qmin, qmax;
      qrange_of_rows(c.qspans, r0, r1, &qmin, &qmax);
      int owner = 0;
      for (const Span& qs : c.qspans)
        if (r0 >= qs.row0 && r0 < qs.row0 + qs.len) owner = qs.owner;
      int64_t n = 0;
      for (const Span& ks : kv) n += live_tiles(c, ks, qmin, qmax);
      tiles[owner] += 2 * n;
    }
  }
  return ok();
}

ra_status ra_device_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(RA_ERR_CUDA, "stream: %s", cudaGetErrorString(e));
  int code = 0, code_bwd = 0;
  int err = ra::read_and_clear_device_error(&code);
  if (err == cudaSuccess) err = ra::read_and_clear_bwd_error(&code_bwd);
  if (err != cudaSuccess) return cuda_status(err, "reading the device status word");
  if (code == 0) code = code_bwd;
  if (code != 0)
    return fail(RA_ERR_TIMEOUT, "a kernel gave up waiting (code %d): its outputs are invalid",
                code);
  return ok();
}

const char* ra_last_error(void) { return g_msg; }

int32_t ra_version(void) { return RA_VERSION; }

}  // extern "C"
