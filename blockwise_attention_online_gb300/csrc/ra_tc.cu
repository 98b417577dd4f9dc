// bf16 ring-attention forward on the 5th-generation tensor cores (sm_103a).
//
// One persistent kernel runs the whole chunk walk of the ring forward pass
// (exercise page "systems-distributed-ring-attention-online-softmax", task
// statement; "Ring Attention: Distributed Reads with Online Softmax",
// section "A simple forward schedule"; glossary "ring attention", algorithm
// steps (1)-(6)). A work unit is (batch, query head, pair of 128-row query
// tiles). For a unit the CTA visits the key/value chunks in the ring order of
// the unit's query segment and, per 128-row key tile:
//
//   S_t = Q_t K^T                      tcgen05.mma, SMEM x SMEM -> TMEM (fp32)
//   mask (causal / ragged), row max, exp2, row sum      softmax warpgroup t
//   lazy rescale of O_t when the running max grows      (online-softmax merge)
//   O_t += P_t V                       tcgen05.mma, TMEM(P, bf16) x SMEM -> TMEM
//
// m, l stay in registers and O in TMEM for the whole walk; only the final
// O = u / l (or u itself for chunk statistics) goes back to HBM.
//
// The softmax comes in two forms, chosen per launch. The two-pass form reads
// all 128 columns of S once (the row max of unmasked chunks reduced by the
// load itself), keeps them in registers and then computes the exponentials,
// with O rescaled when the max grows by more than 2^8. The one-pass form, for
// packed documents without a causal mask (short, masked units), exponentiates
// each 32-column chunk against the row's reference max, which moves (with O,
// the sums and the P already written rescaled) only when a chunk's max exceeds
// it by more than 2^32. Both are exact softmax; each form measured faster on
// its own kind of workload.
//
// Warp roles (384 threads):
//   warp 0      TMA producer: Q tiles once per unit, then K_j, V_j into a ring
//               of shared-memory stages. The pages overlap the transfer of the
//               next key/value shard with work on the current one (blog, "A
//               simple forward schedule"; glossary "Communication overlap");
//               here that is this multi-stage prefetch with full/empty mbarriers.
//   warp 1      MMA issuer (the warp waits, one elected lane issues) and TMEM
//               owner.
//   warps 2-3   start-up helpers: tensor-map prefetch, and one read of every
//               plan line the other roles' first walks need (those walks read
//               the plan one dependent load after another; cached lines cut
//               the time to the first copy and the first S).
//   warps 4-7   softmax warpgroup for query tile 0 (TMEM lanes 0-127)
//   warps 8-11  softmax warpgroup for query tile 1
// The MMA order S0(j) S1(j) | PV0(j) S0(j+1) PV1(j) S1(j+1) | ... lets the
// tensor core work on one tile while the other tile's softmax runs.
//
// TMEM columns: S0/P0 [0,128), S1/P1 [128,256), O0 [256,256+D), O1 [384,384+D).
// P (bf16, two per column) overwrites the first 64 columns of its S after the
// row has been read; tcgen05.mma operations of one thread execute in order, so
// the next S MMA never overtakes the PV MMA that reads P.
//
// Every mbarrier wait is bounded by a time budget. On expiry the kernel records
// a code in a device status word, tells its other warps to stop, waits for its
// own copies and MMAs in flight, frees TMEM and returns.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <mutex>

#include "ra.h"
#include "ra_plan.h"
#include "ra_ptx.cuh"
#include "ra_wait.cuh"

namespace ra {

// Scratch of ra_ring_attention_noalloc: one fixed array per device, part of
// the library's device image (zero at load, kept until the process exits).
// Host code must not use its name as a pointer: the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[RA_NOALLOC_SCRATCH_BYTES];
// the largest split (one CTA per SM of the widest grid, head_dim 128) fits
static_assert(tc_scratch_bytes(kTcMaxGrid, 128) <= RA_NOALLOC_SCRATCH_BYTES,
              "the fixed scratch array must hold the largest stream-K split");

namespace {

using namespace ptx;

constexpr int kThreads = 384;
constexpr float kNegInf = -__builtin_huge_valf();
// Two-pass softmax (no document mask): O and l are rescaled only when the
// running max (log2 units) grows by more than this, so p = 2^(s - m_ref) stays
// below 2^8.
constexpr float kRescaleLog2 = 8.0f;
// One-pass softmax (packed documents): a row's exponent offset (its reference
// max, log2 units) moves, with O, l and lr rescaled, only when a chunk's max
// exceeds it by more than this: then p = 2^(s - m_ref) <= 2^32, and a sum of
// 2^24 such terms times any |V| below 2^60 stays inside fp32's range.
constexpr float kRefSlackLog2 = 32.0f;

template <int D>
struct Cfg {
  static constexpr int kBoxBytes = 128 * 128;     // 128 rows x 64 bf16 (one swizzle atom wide)
  static constexpr int kBoxes = (D + 63) / 64;    // D = 96: the second box is half zero fill
  static constexpr int kTileBytes = kBoxes * kBoxBytes;  // one 128-row bf16 tile
  static constexpr int kStages = (kBoxes == 2) ? 4 : 8;
  static constexpr int kQOff = 0;
  static constexpr int kKvOff = 2 * kTileBytes;
  static constexpr int kBarOff = kKvOff + kStages * kTileBytes;
  static constexpr int kBarBytes = 256;
  // output staging: 4 KB per softmax warp (32 rows x 128 bytes), 1024-byte
  // aligned (the 128-byte swizzle of the O tensor map repeats every 1024)
  static constexpr int kStageOff = kBarOff + 1024;
  static constexpr int kStageBytes = 8 * 4096;
  static constexpr int kSmemBytes = kStageOff + kStageBytes + 1024;  // + alignment slack
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

// Wait sites, reported in the status word as 0x100 | site.
enum : int {
  kSiteProdQ = 1, kSiteProdKv = 2, kSiteMmaQ = 3, kSiteMmaKv = 4, kSiteMmaP = 5,
  kSiteMmaO = 6, kSiteSoftS = 7, kSiteSoftO = 8, kSiteTest = 10,
  kSitePartial = 11
};

struct Unit {
  int b, hq, hkv, qrow0, qseg, n;
  int lo, hi;  // key positions any row of the unit may see: [lo, hi]
};

// Plan tables live in the plan itself (the common case) or, for problems with
// more chunks or spans than it holds, in device memory; the two are read in
// separate branches (ld_qpiece / ld_kvseg for the device copies).
// Query spans.
__device__ __forceinline__ QPiece qpiece(const TcPlan& p, int i) {
  if (p.ext_qp != nullptr) return ld_qpiece(p.ext_qp + i);
  return p.qp[i];
}

__device__ __forceinline__ int find_piece(const TcPlan& p, int row) {
  int lo = 0, hi = p.n_qpieces - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (qpiece(p, mid).row0 <= row) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ int row_position(const TcPlan& p, int row) {
  const QPiece q = qpiece(p, find_piece(p, row));
  return q.pos0 + q.step * (row - q.row0);
}

// Chunk tables: key spans, the first span of every chunk, tensor maps.
__device__ __forceinline__ KvSeg span_of(const TcPlan& p, int k) {
  if (p.ext_ks != nullptr) return ld_kvseg(p.ext_ks + k);
  return p.ks[k];
}
__device__ __forceinline__ int seg_begin(const TcPlan& p, int c) {
  if (p.ext_csb != nullptr) return __ldg(p.ext_csb + c);
  return p.chunk_seg_begin[c];
}
__device__ __forceinline__ const CUtensorMap* kmap_of(const TcPlan& p, int c) {
  return p.ext_kmap ? p.ext_kmap + c : &p.kmap[c];
}
__device__ __forceinline__ const CUtensorMap* vmap_of(const TcPlan& p, int c) {
  return p.ext_vmap ? p.ext_vmap + c : &p.vmap[c];
}

// Key tiles [tb, te) of span k that hold a position some row of the unit
// may see (not entirely in its future, nor outside its documents).
__device__ __forceinline__ void live_tiles(const TcPlan& p, int k, const Unit& U, int& tb, int& te) {
  const KvSeg s = span_of(p, k);
  if (!p.causal && p.n_docs == 0) {
    tb = 0;
    te = s.ntiles;
    return;
  }
  live_range(s.pos0, s.step, s.len, U.lo, U.hi, tb, te);
}

__device__ __forceinline__ void decode_unit(const TcPlan& p, int u, Unit& U) {
  int rank, ub, uhq;
  unit_coords(u, p.n_qpairs, p.B, p.Hq, p.Hkv, p.pair_block, rank, ub, uhq);
  const int qpair = p.has_order ? int(p.order[rank]) : rank;
  U.b = ub;
  U.hq = uhq;
  U.hkv = U.hq / (p.Hq / p.Hkv);
  U.qrow0 = qpair * kTcRowsPerUnit;
  const int r1 = min(U.qrow0 + kTcRowsPerUnit, p.Sq);
  int i = find_piece(p, U.qrow0);
  U.qseg = qpiece(p, i).seg;
  int qmin = 0x7fffffff, qmax = -1;
  for (; i < p.n_qpieces && qpiece(p, i).row0 < r1; ++i) {
    const QPiece q = qpiece(p, i);
    const int a = max(U.qrow0, q.row0), e = min(r1, q.row0 + q.len);
    qmin = min(qmin, q.pos0 + q.step * (a - q.row0));
    qmax = max(qmax, q.pos0 + q.step * (e - 1 - q.row0));
  }
  // the windows grow with the position: the lowest row bounds lo, the highest hi
  int unused;
  key_window(p, qmin, U.lo, unused);
  key_window(p, qmax, unused, U.hi);
  int n = 0;
  for (int k = 0; k < p.n_kvsegs; ++k) {
    int tb, te;
    live_tiles(p, k, U, tb, te);
    n += te - tb;
  }
  U.n = n;
}

// Walks the live key tiles of a unit: chunks in ring order, spans in order,
// tiles in order. Every warp role runs the same walk. `t` is the tile index
// within the span, `nlive` one past the span's last live tile.
struct TileIter {
  int s, ks, ks_end, t, nlive;
  __device__ __forceinline__ TileIter() : s(-1), ks(0), ks_end(0), t(0), nlive(0) {}
  // Position the walk on tile number `skip` of the unit (whole spans are
  // stepped over at once).
  __device__ __forceinline__ void seek(const TcPlan& p, const Unit& U, int skip) {
    while (skip > 0) {
      if (t < nlive) {
        const int take = min(skip, nlive - t);
        t += take;
        skip -= take;
        continue;
      }
      ++ks;
      if (ks < ks_end) {
        live_tiles(p, ks, U, t, nlive);
        continue;
      }
      if (++s >= p.n_chunks) return;
      const int c = p.ring ? (U.qseg - s + p.n_chunks) % p.n_chunks : s;
      ks = seg_begin(p, c) - 1;
      ks_end = seg_begin(p, c + 1);
      t = 0;
      nlive = 0;
    }
  }
  __device__ __forceinline__ bool next(const TcPlan& p, const Unit& U, int& ks_out, int& t_out) {
    while (true) {
      if (t < nlive) {
        ks_out = ks;
        t_out = t++;
        return true;
      }
      ++ks;
      if (ks < ks_end) {
        live_tiles(p, ks, U, t, nlive);
        continue;
      }
      if (++s >= p.n_chunks) return false;
      const int c = p.ring ? (U.qseg - s + p.n_chunks) % p.n_chunks : s;
      ks = seg_begin(p, c) - 1;
      ks_end = seg_begin(p, c + 1);
      t = 0;
      nlive = 0;
    }
  }
};

// A CTA's work, in order: whole units c, c+G, ... for dp_rounds rounds (in
// odd rounds unit G-1-c instead when the plan says so), then
// its share [sk_bound[c], sk_bound[c+1]) of the key tiles of the remaining
// units laid end to end (a stream-K split; the host places the cuts so that
// shares of tiles plus per-unit fixed costs are equal). A share may begin
// inside a unit (a TAIL part: it publishes
// partial results to its scratch slot) and may end inside one (a HEAD part: it
// merges the partials of the CTAs that hold the rest before the epilogue).
enum : int { kFull = 0, kHead = 1, kTail = 2 };

struct Item {
  int u, t0, t1, kind;
};

struct Walker {
  int k, i;
  long long a, b;
  __device__ __forceinline__ void init(const TcPlan& p) {
    k = 0;
    a = p.sk_bound[blockIdx.x];
    b = p.sk_bound[blockIdx.x + 1];
    i = p.sk_first[blockIdx.x];
  }
  __device__ __forceinline__ bool next(const TcPlan& p, Item& it) {
    if (k < p.dp_rounds) {
      it.u = ((p.dp_snake && (k & 1)) ? p.grid - 1 - int(blockIdx.x) : int(blockIdx.x)) + k * p.grid;
      it.t0 = 0;
      it.t1 = -1;  // the whole unit
      it.kind = kFull;
      ++k;
      return true;
    }
    if (i >= p.sk_units) return false;
    const long long lo = p.sk_prefix[i], hi = p.sk_prefix[i + 1];
    const bool last_cta = int(blockIdx.x) == p.grid - 1;
    if (!(lo < b || (last_cta && lo == b))) return false;
    if (hi <= a && !(hi == lo && lo == a)) return false;  // nothing of it here
    it.u = p.dp_rounds * p.grid + i;
    it.t0 = int((lo > a ? lo : a) - lo);
    it.t1 = int((hi < b ? hi : b) - lo);
    it.kind = (it.t0 > 0) ? kTail : (it.t1 < hi - lo ? kHead : kFull);
    ++i;
    return true;
  }
};

// One warp writes NC 16-byte chunks of each of its 32 output rows (a row piece
// of NC * 16 bytes) through its shared-memory staging area. Each lane deposits
// its own row (chunk slots XOR-swizzled by row, so neither side has bank
// conflicts); then each store instruction covers 32 / NC whole row pieces
// instead of 32 rows 16 bytes apart. Rows at and past `rows_valid` are not
// written. Every lane of the warp must call it.
// One warp writes the 32 rows x 128 bytes of a 64-column O piece through its
// staging area (1024-byte aligned) with one asynchronous TMA store: each
// lane deposits its row in the O map's 128-byte swizzle (16-byte chunk k of
// row r at slot k ^ (r & 7)), and lane 0 issues the copy. The area is
// rewritten only after the warp's previous copy has read it. Rows past the
// end of the sequence are clipped by the map.
__device__ __forceinline__ void warp_store_tma(uint8_t* stage, uint32_t stage_s, const uint4 (&ch)[8],
                                               int lane, const CUtensorMap* omap, int col, int row,
                                               int hq, int b) {
  if (lane == 0) bulk_wait_read_all();
  __syncwarp();
#pragma unroll
  for (int k = 0; k < 8; ++k)
    *reinterpret_cast<uint4*>(stage + lane * 128 + ((k ^ (lane & 7)) * 16)) = ch[k];
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_4d(omap, stage_s, col, row, hq, b);
    bulk_commit_group();
  }
}

template <int NC>
__device__ __forceinline__ void warp_store_staged(uint8_t* stage, const uint4 (&ch)[NC], int lane,
                                                  char* row0, int64_t row_bytes, int rows_valid) {
  static_assert(NC == 4 || NC == 8, "row piece of 64 or 128 bytes");
#pragma unroll
  for (int k = 0; k < NC; ++k)
    *reinterpret_cast<uint4*>(stage + lane * (NC * 16) + ((k ^ (lane & (NC - 1))) * 16)) = ch[k];
  __syncwarp();
  constexpr int kRowsPer = 32 / NC;
  const int kq = lane & (NC - 1), rsub = lane / NC;
#pragma unroll
  for (int it = 0; it < NC; ++it) {
    const int row = it * kRowsPer + rsub;
    const uint4 v =
        *reinterpret_cast<const uint4*>(stage + row * (NC * 16) + ((kq ^ (row & (NC - 1))) * 16));
    if (row < rows_valid) *reinterpret_cast<uint4*>(row0 + row * row_bytes + kq * 16) = v;
  }
  __syncwarp();
}

// Publishing and reading the partial results of split units (global memory,
// release/acquire at GPU scope).
__device__ __forceinline__ void st_release(unsigned* addr, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire(const unsigned* addr) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void wg_bar(int id) {
  asm volatile("bar.sync %0, 128;" ::"r"(id) : "memory");
}

// Rare path of the softmax: O (D fp32 columns at tO) times alpha.
template <int D>
__device__ __noinline__ void rescale_o(uint32_t tO, float alpha) {
#pragma unroll 1
  for (int cc = 0; cc < D / 16; ++cc) {
    uint32_t o[16];
    tmem_ld16(tO + 16 * cc, o);
    tmem_ld_wait();
    reg_fence(o);
#pragma unroll
    for (int c = 0; c < 16; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
    tmem_st16(tO + 16 * cc, o);
  }
}

// Rare path of the softmax: the first n P chunks (bf16 pairs at tS) times
// alpha, rounded again; returns their sums (the lr accumulators).
__device__ __noinline__ float4 rescale_p(uint32_t tS, int n, float alpha) {
  float racc[4] = {0.f, 0.f, 0.f, 0.f};
  tmem_st_wait();
#pragma unroll 1
  for (int cc = 0; cc < n; ++cc) {
    uint32_t w[16];
    tmem_ld16(tS + 16 * cc, w);
    tmem_ld_wait();
    reg_fence(w);
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const float a = __uint_as_float(w[c] << 16) * alpha;
      const float b = __uint_as_float(w[c] & 0xffff0000u) * alpha;
      w[c] = pack_bf16x2(a, b);
      add_bf16x2_halves(racc[2 * (c & 1)], racc[2 * (c & 1) + 1], w[c]);
    }
    tmem_st16(tS + 16 * cc, w);
  }
  return make_float4(racc[0], racc[1], racc[2], racc[3]);
}

template <int D, bool kOnePass, bool kPoll, bool kFull>
__global__ void __launch_bounds__(kThreads, 1) tc_ring_kernel(const __grid_constant__ TcPlan p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const gbase = smem_raw + (base - raw);
  const uint32_t sQ = base + C::kQOff;
  const uint32_t sKV = base + C::kKvOff;
  const uint32_t bars = base + C::kBarOff;
  const uint32_t b_qfull = bars, b_qempty = bars + 8;
  const uint32_t b_kvfull0 = bars + 16, b_kvempty0 = bars + 16 + 8 * C::kStages;
  const uint32_t b_misc = bars + 16 + 16 * C::kStages;
  const uint32_t b_sfull0 = b_misc, b_pfull0 = b_misc + 16, b_ofull0 = b_misc + 32,
                 b_ofree0 = b_misc + 48, b_done = b_misc + 64;
  const uint32_t b_never = b_misc + 72;  // test hook: nobody arrives on it
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::kBarOff + 16 + 16 * C::kStages + 80);
  volatile int* const abort_flag =
      reinterpret_cast<volatile int*>(gbase + C::kBarOff + 16 + 16 * C::kStages + 84);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned long long budget = p.timeout_ns;

  if (threadIdx.x == 0) {
    mbar_init(b_qfull, 1);
    mbar_init(b_qempty, 1);
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(b_kvfull0 + 8 * s, 1);
      mbar_init(b_kvempty0 + 8 * s, 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(b_sfull0 + 8 * t, 1);
      mbar_init(b_pfull0 + 8 * t, 128);
      mbar_init(b_ofull0 + 8 * t, 1);
      mbar_init(b_ofree0 + 8 * t, 128);
    }
    mbar_init(b_done, 1);
    mbar_init(b_never, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 4) {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 104;\n" ::: "memory");
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {  // one thread waits and issues the copies
      int it = 0, qn = 0, fenced = -1;
      bool ok = true;
      Walker wk;
      wk.init(p);
      Item I;
      while (ok && wk.next(p, I)) {
        Unit U;
        decode_unit(p, I.u, U);
        const int n = (I.t1 < 0 ? U.n : I.t1) - I.t0;
        if (n == 0) continue;
        ok = wait_bar(b_qempty, (qn & 1) ^ 1, abort_flag, budget, kSiteProdQ);
        if (!ok) break;
        {
          mbar_arrive_expect_tx(b_qfull, 2 * C::kTileBytes);
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int bx = 0; bx < C::kBoxes; ++bx)
              tma_load_4d(sQ + t * C::kTileBytes + bx * C::kBoxBytes, &p.qmap, b_qfull, bx * 64,
                          U.qrow0 + 128 * t, U.hq, U.b);
        }
        ++qn;
        TileIter iter;
        iter.seek(p, U, I.t0);
        int ks, t;
        for (int j = 0; ok && j < n && iter.next(p, U, ks, t); ++j) {
          const KvSeg sg = span_of(p, ks);
          const int row = sg.row0 + 128 * t;
          if (p.ext_kmap != nullptr && sg.chunk != fenced) {  // maps copied in from the host
            fence_tmap_acquire(kmap_of(p, sg.chunk));
            fence_tmap_acquire(vmap_of(p, sg.chunk));
            fenced = sg.chunk;
          }
#pragma unroll
          for (int kv = 0; kv < 2; ++kv) {
            const int st = it % C::kStages;
            ok = wait_bar(b_kvempty0 + 8 * st, ((it / C::kStages) & 1) ^ 1, abort_flag, budget,
                        kSiteProdKv);
            if (!ok) break;
            {
              const uint32_t full = b_kvfull0 + 8 * st;
              mbar_arrive_expect_tx(full, C::kTileBytes);
              const CUtensorMap* map = kv == 0 ? kmap_of(p, sg.chunk) : vmap_of(p, sg.chunk);
#pragma unroll
              for (int bx = 0; bx < C::kBoxes; ++bx)
                tma_load_4d(sKV + st * C::kTileBytes + bx * C::kBoxBytes, map, full, bx * 64, row,
                            U.hkv, U.b);
            }
            ++it;
          }
        }
      }
      if (!ok) {
        // let the copies already in flight land before the CTA goes away
        for (int s = 0; s < C::kStages; ++s) {
          const int back = ((it - 1 - s) % C::kStages + C::kStages) % C::kStages;
          const int last = it - 1 - back;
          if (last >= 0) drain_wait(b_kvfull0 + 8 * s, (last / C::kStages) & 1, budget);
        }
        if (qn > 0) drain_wait(b_qfull, (qn - 1) & 1, budget);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t kIdQK = idesc_bf16_f32(128, 128, 0, 0);
    constexpr uint32_t kIdPV = idesc_bf16_f32(128, D, 0, 1);
    const uint32_t tS0 = tmem, tO0 = tmem + 256;
    // descriptor start addresses advance in 16-byte units inside the low word
    auto issue_qk = [&](int t, int st) {
      const uint64_t qd = sdesc_sw128(sQ + t * C::kTileBytes, 16, 1024);
      const uint64_t kd = sdesc_sw128(sKV + st * C::kTileBytes, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = uint64_t(((kk >> 2) * C::kBoxBytes + (kk & 3) * 32) >> 4);
        mma_ss(tS0 + 128 * t, qd + off, kd + off, kIdQK, kk > 0 ? 1u : 0u);
      }
    };
    auto issue_pv = [&](int t, int st, bool acc) {
      const uint64_t vd = sdesc_sw128(sKV + st * C::kTileBytes, C::kBoxBytes, 1024);
#pragma unroll
      for (int kk = 0; kk < 128 / 16; ++kk) {
        mma_ts(tO0 + 128 * t, tS0 + 128 * t + kk * 8, vd + uint64_t((kk * 16 * 128) >> 4), kIdPV,
               (acc || kk > 0) ? 1u : 0u);
      }
    };
    // The whole warp runs the walk and the waits, so every descriptor and
    // address stays warp-uniform; one elected lane issues each group of MMAs.
    // (Issuing from a single-lane branch measured 80-110 cycles per MMA, above
    // the 64 cycles an M=128, N=128, K=16 MMA takes.) Per ring step PV_0 goes
    // out as soon as V_j and P_0 are there; the next K tile, whose copy can
    // still be in flight then, is waited for only before the next S, which
    // queues behind PV_0.
    //
    // With kPoll (two-pass form only) the warp polls its barriers instead of
    // sleeping in try_wait: it then reacts to a landed K/V tile or a finished
    // P at once (8K non-causal +2.6%, 32K and 128K causal +2-4%). With packed
    // documents (one-pass form) the polls' issue slots, taken from the
    // softmax warps of the same scheduler, cost as much as they save, and the
    // host leaves polling off for launches of very long units too. The choice
    // is a template parameter: as a runtime branch between the two inlined
    // waits it cost 7% at 8K in the generated code alone.
    static_assert(!(kOnePass && (kPoll || kFull)), "the one-pass form neither polls nor skips the walk");
    auto mwait = [&](uint32_t bar, uint32_t parity, int site) {
      if constexpr (kPoll) return warp_wait_spin(bar, parity, abort_flag, budget, site);
      else return warp_wait(bar, parity, abort_flag, budget, site);
    };
    {
      const bool leader = elect_one();
      int it = 0, qn = 0, un = 0;
      uint32_t pc0 = 0, pc1 = 0;
      bool ok = true;
      if (p.test_stall) ok = warp_wait(b_never, 0, abort_flag, budget, kSiteTest);
      Walker wk;
      wk.init(p);
      Item I;
      while (ok && wk.next(p, I)) {
        Unit U;
        decode_unit(p, I.u, U);
        const int n = (I.t1 < 0 ? U.n : I.t1) - I.t0;
        if (n == 0) continue;
        ok = mwait(b_qfull, qn & 1, kSiteMmaQ);
        if (!ok) break;
        ++qn;
        int kst = it % C::kStages;
        ok = mwait(b_kvfull0 + 8 * kst, (it / C::kStages) & 1, kSiteMmaKv);
        if (!ok) break;
        ++it;
        tc_fence_after();
        if (leader) {
          issue_qk(0, kst);
          mma_commit(b_sfull0);
          issue_qk(1, kst);
          mma_commit(b_sfull0 + 8);
          mma_commit(b_kvempty0 + 8 * kst);
          if (n == 1) mma_commit(b_qempty);
        }
        __syncwarp();
        for (int j = 0; j < n; ++j) {
          const bool more = j + 1 < n;
          const int vst = it % C::kStages;
          ok = mwait(b_kvfull0 + 8 * vst, (it / C::kStages) & 1, kSiteMmaKv);
          if (!ok) break;
          ++it;
          // query tile 0: PV as soon as P_0 is there, then (once the next K
          // tile has landed) the next S behind it in the same queue
          ok = mwait(b_pfull0, pc0 & 1, kSiteMmaP);
          if (!ok) break;
          ++pc0;
          if (j == 0) {
            ok = mwait(b_ofree0, (un & 1) ^ 1, kSiteMmaO);
            if (!ok) break;
          }
          tc_fence_after();
          if (leader) {
            issue_pv(0, vst, j > 0);
            if (!more) mma_commit(b_ofull0);
          }
          __syncwarp();
          if (more) {
            kst = it % C::kStages;
            ok = mwait(b_kvfull0 + 8 * kst, (it / C::kStages) & 1, kSiteMmaKv);
            if (!ok) break;
            ++it;
            tc_fence_after();
            if (leader) {
              issue_qk(0, kst);
              mma_commit(b_sfull0);
            }
            __syncwarp();
          }
          // query tile 1
          ok = mwait(b_pfull0 + 8, pc1 & 1, kSiteMmaP);
          if (!ok) break;
          ++pc1;
          if (j == 0) {
            ok = mwait(b_ofree0 + 8, (un & 1) ^ 1, kSiteMmaO);
            if (!ok) break;
          }
          tc_fence_after();
          if (leader) {
            issue_pv(1, vst, j > 0);
            mma_commit(b_kvempty0 + 8 * vst);
            if (!more) mma_commit(b_ofull0 + 8);
            if (more) {
              issue_qk(1, kst);
              mma_commit(b_sfull0 + 8);
              mma_commit(b_kvempty0 + 8 * kst);
              if (j + 2 == n) mma_commit(b_qempty);
            }
          }
          __syncwarp();
        }
        ++un;
      }
      // every MMA this warp issued must be complete before TMEM is freed
      if (leader) mma_commit(b_done);
      __syncwarp();
      drain_wait(b_done, 0, budget);
    }
    __syncwarp();
  } else if (warp == 2) {
    // tensor maps into the TMA unit's cache ahead of their first copies, one
    // lane per chunk (the chunk-table reads overlap)
    if (lane == 0) prefetch_tmap(&p.qmap);
    if (p.ext_kmap == nullptr) {
#pragma unroll
      for (int k = 0; k < kTcMaxChunks / 32; ++k) {
        const int c = lane + 32 * k;
        if (c < p.n_chunks && p.chunk_seg_begin[c] != p.chunk_seg_begin[c + 1]) {
          prefetch_tmap(&p.kmap[c]);
          prefetch_tmap(&p.vmap[c]);
        }
      }
    }
  } else {
    // warp 3: the plan lines that the first walks of the other roles read one
    // after another, read here all at once so that those reads hit
    uint32_t v[12];
    v[0] = uint32_t(p.sk_prefix[min(lane * 16, min(p.sk_units, kTcMaxSkUnits))]);
    v[1] = uint32_t(p.sk_bound[min(lane * 16, min(p.grid, kTcMaxGrid))]);
    v[2] = uint32_t(p.sk_first[max(0, min(lane * 32, min(p.grid, kTcMaxGrid) - 1))]);
    v[3] = uint32_t(p.chunk_seg_begin[min(lane * 16, min(p.n_chunks, kTcMaxChunks))]);
    v[4] = uint32_t(p.qp[min(lane, kMaxQPieces - 1)].row0);
    v[5] = uint32_t(p.qp[min(lane + 32, kMaxQPieces - 1)].row0);
    v[6] = uint32_t(p.ks[min(lane, kTcMaxKvSegs - 1)].ntiles);
    v[7] = uint32_t(p.ks[min(lane + 32, kTcMaxKvSegs - 1)].ntiles);
    v[8] = uint32_t(p.doc_bounds[min(lane * 16, min(p.n_docs, kMaxDocs))]);
    v[9] = uint32_t(p.doc_bounds[min(lane * 16 + 512, min(p.n_docs, kMaxDocs))]);
    v[10] = uint32_t(p.B + p.Hq + p.n_qpieces + p.dp_rounds);
    v[11] = uint32_t(p.ext_ks != nullptr) + uint32_t(p.n_units);
    uint32_t acc = 0;
#pragma unroll
    for (int i = 0; i < 12; ++i) acc ^= v[i];
    asm volatile("" ::"r"(acc));
  }
  } else {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 200;\n" ::: "memory");
    // ------------------------------------------------------------ softmax
    const int wg = (warp - 4) >> 2;
    const int sub = warp & 3;
    const int r = sub * 32 + lane;
    const uint32_t lane_off = uint32_t(sub * 32) << 16;
    const uint32_t tS = tmem + wg * 128 + lane_off;
    const uint32_t tO = tmem + 256 + wg * 128 + lane_off;
    const uint32_t b_sfull = b_sfull0 + 8 * wg, b_pfull = b_pfull0 + 8 * wg;
    const uint32_t b_ofull = b_ofull0 + 8 * wg, b_ofree = b_ofree0 + 8 * wg;
    const float c2 = p.scale_log2;
    uint32_t sc = 0, oc = 0;
    bool ok = true;
    Walker wk;
    wk.init(p);
    Item I;
    while (ok && wk.next(p, I)) {
      Unit U;
      decode_unit(p, I.u, U);
      const int n = (I.t1 < 0 ? U.n : I.t1) - I.t0;
      const int grow = U.qrow0 + wg * 128 + r;
      const bool rvalid = grow < p.Sq;
      // keys this row may see: positions [rlo, rhi]
      int rlo = 0, rhi = 0x7ffffffe;
      if (rvalid && (p.causal || p.n_docs > 0)) key_window(p, row_position(p, grow), rlo, rhi);
      float m_ref = kNegInf, mx = kNegInf, l = 0.f, lr = 0.f;
      // Launches whose key tiles are all whole and visible to every row
      // (kFull, chosen by the host from full_tiles) skip the walk over the
      // key spans: its dependent plan reads sat between a step's P and the
      // next S (8K +2.3%; as a runtime flag only +1%).
      constexpr bool walk = !kFull;
      if (n > 0) {
        TileIter iter;
        if (walk) iter.seek(p, U, I.t0);
        int ks = 0, t = 0, sg_k = -1;
        KvSeg sg = {};
        for (int j = 0; j < n; ++j) {
          // visible columns of this row: the range [C0, L) of the tile (known
          // before S arrives; C0 > 0 only where a document starts inside it)
          int L = 128, C0 = 0;
          if (walk) {
            if (!iter.next(p, U, ks, t)) break;
            if (ks != sg_k) {  // the span's fields stay in registers while its tiles run
              sg = span_of(p, ks);
              sg_k = ks;
            }
            L = min(128, sg.len - 128 * t);
            if (p.causal || p.n_docs) {
              const int first = sg.pos0 + sg.step * (128 * t);
              if (sg.step == 1) {
                L = rhi < first ? 0 : min(L, rhi - first + 1);
                if (rlo > first) C0 = min(L, rlo - first);
              } else {
                L = rhi < first ? 0 : min(L, (rhi - first) / sg.step + 1);
                if (rlo > first) C0 = min(L, (rlo - first - 1) / sg.step + 1);
              }
            }
          }
          ok = warp_wait(b_sfull, sc & 1, abort_flag, budget, kSiteSoftS);
          if (!ok) break;
          ++sc;
          tc_fence_after();
          if constexpr (kOnePass) {
            // One pass over S in 32-column chunks. The exponent offset is the
            // row's reference max m_ref (log2 units): set from the max of the
            // row's first visible chunk and moved only when a chunk's max exceeds
            // it by more than kRefSlackLog2, so p = 2^(s*c2 - m_ref) stays below
            // 2^kRefSlackLog2 (far from overflow; floating point is scale
            // invariant, and O, l, lr carry the same scale). Each chunk's max is
            // reduced first, as a shallow tree; a chunk that moves the reference
            // first rescales O, the sums and this step's P chunks already
            // written (warp-uniform, since TMEM access is warp-collective; rows
            // that keep their reference take alpha = 1).
            const uint64_t c2x2 = f2(c2, c2);
            uint64_t lacc[2] = {0, 0};
            float racc[4] = {0.f, 0.f, 0.f, 0.f};
            float rmax = kNegInf;
  #pragma unroll 1
            for (int i = 0; i < 4; ++i) {
              uint32_t s[32];
              float cm;
              if (__any_sync(0xffffffffu, L < 32 * i + 32 || C0 > 32 * i)) {
                // some row of this warp has masked columns in the chunk
                tmem_ld32(tS + 32 * i, s);
                tmem_ld_wait();
                reg_fence(s);
  #pragma unroll
                for (int c = 0; c < 32; ++c)
                  if (32 * i + c >= L || 32 * i + c < C0) s[c] = 0xff800000u;  // -inf
                float t[8];
  #pragma unroll
                for (int a = 0; a < 8; ++a)
                  t[a] = max3(__uint_as_float(s[4 * a]), __uint_as_float(s[4 * a + 1]),
                              fmaxf(__uint_as_float(s[4 * a + 2]), __uint_as_float(s[4 * a + 3])));
                cm = max3(max3(t[0], t[1], t[2]), max3(t[3], t[4], t[5]), fmaxf(t[6], t[7]));
              } else {
                // nothing masked: the load reduces the chunk to its max on the way
                tmem_ld32_max(tS + 32 * i, s, cm);
                tmem_ld_wait();
                reg_fence(s);
                asm volatile("" : "+f"(cm));
              }
              rmax = fmaxf(rmax, cm);
              const bool move = cm * c2 > m_ref + kRefSlackLog2;  // any finite cm when m_ref = -inf
              if (__any_sync(0xffffffffu, move)) {
                const float m_to = move ? cm * c2 : m_ref;
                const float alpha = move ? ex2(m_ref - m_to) : 1.f;  // 0 from -inf
                l *= alpha;
                lr *= alpha;
                if (j > 0) rescale_o<D>(tO, alpha);
                float a0, a1, a2, a3;
                f2_split(lacc[0], a0, a1);
                f2_split(lacc[1], a2, a3);
                lacc[0] = f2(a0 * alpha, a1 * alpha);
                lacc[1] = f2(a2 * alpha, a3 * alpha);
                const float4 rs = rescale_p(tS, i, alpha);
                racc[0] = rs.x;
                racc[1] = rs.y;
                racc[2] = rs.z;
                racc[3] = rs.w;
                m_ref = m_to;
              }
              const float off = (m_ref == kNegInf) ? 0.f : m_ref;
              const uint64_t noff = f2(-off, -off);
              uint32_t pk[16];
  #pragma unroll
              for (int c = 0; c < 16; ++c) {
                float x0, x1;
                f2_split(fma2(f2(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])), c2x2, noff),
                         x0, x1);
                const float a = ex2(x0), b = ex2(x1);
                lacc[c & 1] = add2(lacc[c & 1], f2(a, b));
                const uint32_t w = pack_bf16x2(a, b);
                add_bf16x2_halves(racc[2 * (c & 1)], racc[2 * (c & 1) + 1], w);
                pk[c] = w;
              }
              tmem_st16(tS + 16 * i, pk);
            }
            mx = fmaxf(mx, rmax);
            {
              float a0, a1, a2, a3;
              f2_split(lacc[0], a0, a1);
              f2_split(lacc[1], a2, a3);
              l += (a0 + a1) + (a2 + a3);
              lr += (racc[0] + racc[1]) + (racc[2] + racc[3]);
            }
          } else {
            // Pass 1: row max. All 128 columns are read with a single wait (the
            // load latency is paid once) and stay in registers; pass 2 turns
            // them into P chunk by chunk without reading S again.
            float mx0 = kNegInf, mx1 = kNegInf;
            uint32_t s[4][32];  // the row's scores, kept for pass 2
            if (__any_sync(0xffffffffu, L < 128 || C0 > 0)) {
              // some row of this warp has masked columns: mask, then reduce
  #pragma unroll
              for (int i = 0; i < 4; ++i) tmem_ld32(tS + 32 * i, s[i]);
              tmem_ld_wait();
  #pragma unroll
              for (int i = 0; i < 4; ++i) reg_fence(s[i]);
              if (L < 128 || C0 > 0) {
  #pragma unroll
                for (int i = 0; i < 4; ++i)
  #pragma unroll
                  for (int c = 0; c < 32; ++c)
                    if (32 * i + c >= L || 32 * i + c < C0) s[i][c] = 0xff800000u;  // -inf
              }
  #pragma unroll
              for (int i = 0; i < 4; ++i)
  #pragma unroll
                for (int c = 0; c < 32; c += 4) {
                  mx0 = max3(mx0, __uint_as_float(s[i][c]), __uint_as_float(s[i][c + 1]));
                  mx1 = max3(mx1, __uint_as_float(s[i][c + 2]), __uint_as_float(s[i][c + 3]));
                }
            } else {
              // nothing masked: the tensor-memory loads reduce each 32-column
              // chunk to its max on the way (the values themselves are not
              // needed in this pass)
              float m4[4];
  #pragma unroll
              for (int i = 0; i < 4; ++i) tmem_ld32_max(tS + 32 * i, s[i], m4[i]);
              tmem_ld_wait();
  #pragma unroll
              for (int i = 0; i < 4; ++i) {
                reg_fence(s[i]);
                asm volatile("" : "+f"(m4[i]));
              }
              mx0 = fmaxf(m4[0], m4[1]);
              mx1 = fmaxf(m4[2], m4[3]);
            }
            const float rmax = fmaxf(mx0, mx1);
            mx = fmaxf(mx, rmax);
            const float mnew = rmax * c2;
            // The O rescale touches TMEM with warp-collective loads and stores, so
            // the whole warp takes the branch when any of its rows needs it; rows
            // that do not need it keep their reference max (alpha = 1).
            const bool grow_ref = mnew > m_ref + kRescaleLog2;
            if (__any_sync(0xffffffffu, grow_ref)) {
              const float m_to = grow_ref ? mnew : m_ref;
              const float alpha = grow_ref ? ex2(m_ref - mnew) : 1.f;
              l *= alpha;
              lr *= alpha;
              if (j > 0) {
  #pragma unroll 1
                for (int cc = 0; cc < D / 16; ++cc) {
                  uint32_t o[16];
                  tmem_ld16(tO + 16 * cc, o);
                  tmem_ld_wait();
                  reg_fence(o);
  #pragma unroll
                  for (int c = 0; c < 16; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
                  tmem_st16(tO + 16 * cc, o);
                }
              }
              m_ref = m_to;
            }
            const float off = (m_ref == kNegInf) ? 0.f : m_ref;
            // p = 2^(s*c2 - off) two at a time; l sums the fp32 p (returned), lr
            // sums the bf16-rounded p that P.V actually uses (normalises O)
            const uint64_t c2x2 = f2(c2, c2), noff = f2(-off, -off);
            uint64_t lacc[2] = {0, 0};
            float racc[4] = {0.f, 0.f, 0.f, 0.f};
            // Pass 2: S chunk i (columns 32i.., in registers) -> P columns 16i..
  #pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint32_t pk[16];
  #pragma unroll
              for (int c = 0; c < 16; ++c) {
                float x0, x1;
                f2_split(fma2(f2(__uint_as_float(s[i][2 * c]), __uint_as_float(s[i][2 * c + 1])), c2x2, noff),
                         x0, x1);
                const float a = ex2(x0), b = ex2(x1);
                lacc[c & 1] = add2(lacc[c & 1], f2(a, b));
                const uint32_t w = pack_bf16x2(a, b);
                add_bf16x2_halves(racc[2 * (c & 1)], racc[2 * (c & 1) + 1], w);
                pk[c] = w;
              }
              tmem_st16(tS + 16 * i, pk);
            }
            {
              float a0, a1, a2, a3;
              f2_split(lacc[0], a0, a1);
              f2_split(lacc[1], a2, a3);
              l += (a0 + a1) + (a2 + a3);
              lr += (racc[0] + racc[1]) + (racc[2] + racc[3]);
            }
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(b_pfull);
        }
        if (!ok) break;
        ok = warp_wait(b_ofull, oc & 1, abort_flag, budget, kSiteSoftO);
        if (!ok) break;
        ++oc;
        tc_fence_after();
      }
      // O is read and written in kParts parts of kHalf 32-column chunks: two
      // halves when D is a multiple of 64, else one 32-column chunk per part
      constexpr int kParts = (D % 64 == 0) ? 2 : D / 32;
      constexpr int kHalf = D / 32 / kParts;
      const size_t slot_row = (size_t(blockIdx.x) * 2 + wg) * 128 + r;
      // A scratch slot (one per CTA and warpgroup) holds raw O as [D/4][128]
      // float4: lane r touches element (k, r), so every warp access covers
      // 512 contiguous bytes.
      constexpr size_t kSlotF4 = size_t(128) * (D / 4);
      if (I.kind == kTail) {
        // ---- publish this part's raw partial results for the unit's head
        float4* const dst = reinterpret_cast<float4*>(p.scratch.o) + (size_t(blockIdx.x) * 2 + wg) * kSlotF4 + r;
#pragma unroll
        for (int h = 0; h < kParts; ++h) {
          uint32_t o[kHalf][32];
#pragma unroll
          for (int cc = 0; cc < kHalf; ++cc) tmem_ld32(tO + 32 * (h * kHalf + cc), o[cc]);
          tmem_ld_wait();
#pragma unroll
          for (int cc = 0; cc < kHalf; ++cc) reg_fence(o[cc]);
          if (h == kParts - 1) {
            tc_fence_before();
            mbar_arrive(b_ofree);
          }
#pragma unroll
          for (int cc = 0; cc < kHalf; ++cc)
#pragma unroll
            for (int c = 0; c < 32; c += 4)
              dst[size_t((h * kHalf * 32 + cc * 32 + c) / 4) * 128] =
                  make_float4(__uint_as_float(o[cc][c]), __uint_as_float(o[cc][c + 1]),
                              __uint_as_float(o[cc][c + 2]), __uint_as_float(o[cc][c + 3]));
        }
        p.scratch.stats[slot_row] = make_float4(m_ref, mx, l, lr);
        wg_bar(1 + wg);
        if (r == 0) {
          __threadfence();
          st_release(p.scratch.flags + blockIdx.x * 2 + wg, p.epoch);
        }
        continue;
      }
      // ---- a head part: merge the partials of the CTAs holding the unit's rest
      float a_self = 1.f;
      int c_first = 0, c_end = 0;  // CTAs [c_first, c_end) hold later parts
      if (I.kind == kHead) {
        const int hi = p.sk_prefix[I.u - p.dp_rounds * p.grid + 1];
        c_first = blockIdx.x + 1;
        c_end = c_first;
        while (c_end < p.grid && p.sk_bound[c_end] < hi) ++c_end;
        // wait for every later part's flag (one thread polls, the warpgroup follows)
        if (r == 0) {
          for (int c = c_first; c < c_end; ++c) {
            if (p.sk_bound[c] >= p.sk_bound[c + 1]) continue;  // that CTA holds no tiles at all
            const unsigned* f = p.scratch.flags + c * 2 + wg;
            unsigned long long t0 = 0;
            for (uint32_t k = 1; ld_acquire(f) != p.epoch; ++k) {
              if ((k & 255u) == 0) {
                if (*abort_flag) break;
                const unsigned long long now = globaltimer();
                if (t0 == 0) t0 = now;
                else if (now - t0 > budget) {
                  *abort_flag = 1;
                  record_error(0x100 | kSitePartial);
                  break;
                }
              }
            }
          }
        }
        wg_bar(1 + wg);
        if (__any_sync(0xffffffffu, *abort_flag != 0)) {  // warp-uniform: TMEM loads follow
          ok = false;
          // TMEM O must still be released for the MMA warp's bookkeeping
          if (n > 0) {
            tc_fence_before();
            mbar_arrive(b_ofree);
          }
          break;
        }
        float M = m_ref;
        for (int c = c_first; c < c_end; ++c) {
          if (p.sk_bound[c] >= p.sk_bound[c + 1]) continue;
          const float4 st = __ldcg(p.scratch.stats + (size_t(c) * 2 + wg) * 128 + r);
          M = fmaxf(M, st.x);
        }
        a_self = (m_ref == kNegInf) ? 0.f : ex2(m_ref - M);
        l *= a_self;
        lr *= a_self;
        for (int c = c_first; c < c_end; ++c) {
          if (p.sk_bound[c] >= p.sk_bound[c + 1]) continue;
          const float4 st = __ldcg(p.scratch.stats + (size_t(c) * 2 + wg) * 128 + r);
          const float bp = (st.x == kNegInf) ? 0.f : ex2(st.x - M);
          mx = fmaxf(mx, st.y);
          l += bp * st.z;
          lr += bp * st.w;
        }
        m_ref = M;
      }
      // epilogue: read O in halves (bounded register use), fold in any
      // partials, release TMEM after the last read, write this row's results
      const bool any = mx != kNegInf;
      const float corr = any ? ex2(m_ref - mx * c2) : 0.f;
      const float fo = p.stats_mode ? corr * (lr > 0.f ? l / lr : 0.f) : (lr > 0.f ? 1.f / lr : 0.f);
      // this warp's 32 output rows start at row wrow0; rows past Sq are not written
      const int wrow0 = U.qrow0 + wg * 128 + sub * 32;
      const int wvalid = min(32, max(0, p.Sq - wrow0));
      const int64_t wbase = int64_t(U.b) * p.o_sb + int64_t(U.hq) * p.o_sh + int64_t(wrow0) * p.o_sr;
      uint8_t* const stage = gbase + C::kStageOff + (warp - 4) * 4096;
#pragma unroll
      for (int h = 0; h < kParts; ++h) {
        uint32_t o[kHalf][32];
        if (n > 0) {
#pragma unroll
          for (int cc = 0; cc < kHalf; ++cc) tmem_ld32(tO + 32 * (h * kHalf + cc), o[cc]);
          tmem_ld_wait();
#pragma unroll
          for (int cc = 0; cc < kHalf; ++cc) reg_fence(o[cc]);
          if (h == kParts - 1) {
            tc_fence_before();
            mbar_arrive(b_ofree);
          }
        } else {
#pragma unroll
          for (int cc = 0; cc < kHalf; ++cc)
#pragma unroll
            for (int c = 0; c < 32; ++c) o[cc][c] = 0u;
        }
        if (I.kind == kHead) {
#pragma unroll
          for (int cc = 0; cc < kHalf; ++cc)
#pragma unroll
            for (int c = 0; c < 32; ++c) o[cc][c] = __float_as_uint(__uint_as_float(o[cc][c]) * a_self);
          for (int c = c_first; c < c_end; ++c) {
            if (p.sk_bound[c] >= p.sk_bound[c + 1]) continue;
            const size_t prow = (size_t(c) * 2 + wg) * 128 + r;
            const float4 st = __ldcg(p.scratch.stats + prow);
            const float bp = (st.x == kNegInf) ? 0.f : ex2(st.x - m_ref);
            const float4* src = reinterpret_cast<const float4*>(p.scratch.o) + (size_t(c) * 2 + wg) * kSlotF4 + r;
#pragma unroll
            for (int cc = 0; cc < kHalf; ++cc)
#pragma unroll
              for (int c4 = 0; c4 < 32; c4 += 4) {
                const float4 v = __ldcg(src + size_t((h * kHalf * 32 + cc * 32 + c4) / 4) * 128);
                o[cc][c4] = __float_as_uint(fmaf(bp, v.x, __uint_as_float(o[cc][c4])));
                o[cc][c4 + 1] = __float_as_uint(fmaf(bp, v.y, __uint_as_float(o[cc][c4 + 1])));
                o[cc][c4 + 2] = __float_as_uint(fmaf(bp, v.z, __uint_as_float(o[cc][c4 + 2])));
                o[cc][c4 + 3] = __float_as_uint(fmaf(bp, v.w, __uint_as_float(o[cc][c4 + 3])));
              }
          }
        }
        // write this half through the warp's staging area: a TMA store of the
        // staged rows (bf16 O, head_dim 128) or whole-row stores by the warp
        if (p.o_fp32) {
#pragma unroll
          for (int cc = 0; cc < kHalf; ++cc) {
            uint4 ch[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              ch[k] = make_uint4(__float_as_uint(__uint_as_float(o[cc][4 * k]) * fo),
                                 __float_as_uint(__uint_as_float(o[cc][4 * k + 1]) * fo),
                                 __float_as_uint(__uint_as_float(o[cc][4 * k + 2]) * fo),
                                 __float_as_uint(__uint_as_float(o[cc][4 * k + 3]) * fo));
            warp_store_staged<8>(stage, ch, lane,
                                 reinterpret_cast<char*>(static_cast<float*>(p.out) + wbase + h * kHalf * 32 + cc * 32),
                                 p.o_sr * 4, wvalid);
          }
        } else {
          constexpr int NC = kHalf * 4;
          uint4 ch[NC];
#pragma unroll
          for (int k = 0; k < NC; ++k) {
            const int cc = k >> 2, c = (k & 3) * 8;
            ch[k].x = pack_bf16x2(__uint_as_float(o[cc][c]) * fo, __uint_as_float(o[cc][c + 1]) * fo);
            ch[k].y = pack_bf16x2(__uint_as_float(o[cc][c + 2]) * fo, __uint_as_float(o[cc][c + 3]) * fo);
            ch[k].z = pack_bf16x2(__uint_as_float(o[cc][c + 4]) * fo, __uint_as_float(o[cc][c + 5]) * fo);
            ch[k].w = pack_bf16x2(__uint_as_float(o[cc][c + 6]) * fo, __uint_as_float(o[cc][c + 7]) * fo);
          }
          if constexpr (NC == 8) {
            if (p.o_tma) {
              if (wvalid > 0)
                warp_store_tma(stage, smem_addr(stage), ch, lane, &p.omap, h * 64, wrow0, U.hq, U.b);
              continue;
            }
          }
          warp_store_staged<NC>(stage, ch, lane,
                                reinterpret_cast<char*>(static_cast<uint16_t*>(p.out) + wbase + h * kHalf * 32),
                                p.o_sr * 2, wvalid);
        }
      }
      if (rvalid) {
        const size_t ml_idx = (size_t(U.b) * p.Hq + U.hq) * size_t(p.Sq) + grow;
        p.m[ml_idx] = mx * p.scale;
        p.l[ml_idx] = l * corr;
      }
    }
    // this warp's O copies are complete before its staging area goes away
    if (lane == 0) bulk_wait_all();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

void tc_scratch_carve(void* base, int grid, int D, TcScratch* s) {
  char* b = static_cast<char*>(base);
  s->o = reinterpret_cast<float*>(b);
  b += size_t(grid) * 2 * 128 * D * 4;
  s->stats = reinterpret_cast<float4*>(b);
  b += size_t(grid) * 2 * 128 * 16;
  s->flags = reinterpret_cast<unsigned*>(b);
}

template <int D, bool kOnePass, bool kPoll, bool kFull>
static int launch_d(const TcPlan& plan, void* stream) {
  cudaError_t e = cudaFuncSetAttribute(tc_ring_kernel<D, kOnePass, kPoll, kFull>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(plan.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg<D>::kSmemBytes;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  // a head part waits for partials of later CTAs: all CTAs must be resident
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = plan.scratch.flags != nullptr ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, tc_ring_kernel<D, kOnePass, kPoll, kFull>, plan);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// The kernel instance for a plan: the softmax form, the MMA warp's wait mode
// and whether the softmax warps walk the key spans (all compile-time choices:
// as runtime branches they cost several percent in the generated code).
template <int D>
static int launch_for(const TcPlan& plan, bool one, void* stream) {
  if (one) return launch_d<D, true, false, false>(plan, stream);
  const bool poll = plan.mma_poll != 0, full = plan.full_tiles != 0;
  if (full)
    return poll ? launch_d<D, false, true, true>(plan, stream) : launch_d<D, false, false, true>(plan, stream);
  return poll ? launch_d<D, false, true, false>(plan, stream) : launch_d<D, false, false, false>(plan, stream);
}

int launch_tc_bf16(const TcPlan& plan, int D, void* stream) {
  if (plan.grid <= 0) return cudaSuccess;
  // packed documents without a causal mask: the one-pass softmax (short,
  // masked units; measured faster there); otherwise the two-pass one (also
  // faster with documents under a causal mask, where units are longer)
  const bool one = plan.n_docs > 0 && !plan.causal;
  switch (D) {
    case 128: return launch_for<128>(plan, one, stream);
    case 96: return launch_for<96>(plan, one, stream);
    default: return launch_for<64>(plan, one, stream);
  }
}

// Unique id of the calling thread's current CUDA context (0 if none is
// current or the driver cannot say). Context ids are never reused within a
// process, so a device reset, which replaces the primary context, changes it.
static unsigned long long current_context_id() {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// The array's device address in the current context. The lookup runs once
// per device and context (with that device current); a cached address is
// reused only while the same context is current, so a device reset leads to
// a fresh lookup instead of a stale pointer.
int tc_static_scratch(void** ptr, size_t* bytes) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  static unsigned long long ctx_of[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  const unsigned long long ctx = current_context_id();
  if (addr[dev] == nullptr || ctx == 0 || ctx != ctx_of[dev]) {
    void* a = nullptr;
    e = cudaGetSymbolAddress(&a, g_noalloc_scratch);  // makes the context current if needed
    if (e != cudaSuccess) return e;
    addr[dev] = a;
    ctx_of[dev] = current_context_id();
  }
  *ptr = addr[dev];
  *bytes = sizeof(g_noalloc_scratch);
  return cudaSuccess;
}

int read_and_clear_device_error(int* code) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_ra_device_error, sizeof(int));
  if (e != cudaSuccess) return e;
  *code = v;
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_ra_device_error, &zero, sizeof(int));
  }
  return e;
}

}  // namespace ra
