// attn_fwd.cu -- fused relative-position attention forward for sm_103a.
//
// Persistent kernel: one CTA per SM walks a list of work items. An item is
// a pair of 128-row query tiles (a and b) of one (batch, head); both tiles
// share one stream of 128-key K/V tiles through shared memory:
//
//   warp 0       TMA producer: the item's two Q tiles and the 3-stage K ring
//                (running ahead into the next item).
//   warp 2       TMA producer of the V ring.
//   warps 1, 3   tcgen05 issuers of tiles a and b (warp 1 also owns TMEM). For
//                each key tile j an issuer computes S = Q K_{j+1}^T as soon as
//                its softmax has read S_j out of TMEM, and O += P_j V_j as soon
//                as P_j is back in TMEM, so the scores of the next key tile are
//                ready when the softmax finishes the current one.
//   warps 4-7    softmax warpgroup of tile a; warps 8-11 that of tile b.
//                Thread t owns query row t (TMEM lane t): it loads its S row
//                from TMEM, adds the relative term, masks, keeps the running
//                max / sum, writes the bf16 probabilities back to TMEM (the
//                A operand of the P.V product) and, at the end of the item,
//                normalises its O row and stores it.
//
// Tensor memory (512 columns): S_a 0-127, S_b 128-255, O_a 256-319,
// O_b 320-383, P_a 384-447, P_b 448-511.
//
// The relative term follows "Relative Position Embeddings, in depth": T5 adds
// a per-head scalar by bucket of the key-minus-query offset ("T5: one scalar
// per head, looked up by bucket"); Shaw adds q_i . a_K[clip(j - i)] to the
// logit and sum_j p_ij a_V[clip(j - i)] to the output ("Shaw et al."). Both
// depend on the offset only, so a tile whose offsets all lie beyond the
// saturation distance needs one constant (T5) or one per-row constant (Shaw)
// instead of per-element lookups; the per-element T5 bias comes from a
// bias-by-offset table in shared memory, read four values per load. DeBERTa
// ("DeBERTa: disentangled content and position") reads, for tiles inside the
// band, the c2p + p2c values its pre-pass wrote per query row and key offset
// (16-byte aligned windows), and beyond the band one saturated c2p value per
// row plus one saturated p2c value per key. ALiBi ("ALiBi and RoPE: the two
// endpoints") needs no table: the slope times the distance is a row constant
// plus a per-column term, exact per column across the diagonal.
//
// Softmax runs in the log2 domain with a lazily updated running maximum: the
// O accumulator in TMEM is rescaled only when a row's maximum grows by more
// than 2^8, which bounds every probability by 256 and is exact because the
// final division uses the same stale maximum.

#include <cuda.h>
#include <cuda_bf16.h>

#include <atomic>
#include <cstdint>

#include "ptx.cuh"
#include "relpos_common.cuh"
#include "relpos_internal.h"

namespace relpos {
namespace {

constexpr int kBM = 128;       // query rows per tile (two tiles per item)
constexpr int kBN = 128;       // keys per tile
constexpr int kStages = 3;     // K/V ring depth (barrier slots; Smem<MODE>::kStages are used)
constexpr int kThreads = 384;  // 12 warps
constexpr uint32_t kTileBytes = kBM * kHeadDim * 2;  // 16 KB: 128 rows x 128 B
// Kernel variants are keyed by MD = mode + 8 for head dimension 128 (T5 and
// ALiBi): MD & 7 is the mode.
__host__ __device__ constexpr int md_mode(int md) { return md & 7; }
__host__ __device__ constexpr int md_dim(int md) { return md >= 8 ? 128 : 64; }
// Shared-memory layout: the item's two query tiles, the K ring, the V ring,
// the barriers, then the mode's tables. Transformer-XL (MODE 4) scores
// against a 128-wide contraction (content and position halves), and at head
// dimension 128 every row is 128 wide: those query tiles and K stages (and
// V stages at d = 128) hold two 64-column halves of kTileBytes each.
template <int MD>
struct Smem {
  static constexpr int MODE = md_mode(MD);
  static constexpr int DH = md_dim(MD);
  // K / V ring depth: Shaw keeps two stages, for the shared memory of its
  // per-row tables (k up to 27); so does d = 128, for its double-size tiles
  static constexpr int kStages = (MODE == 1 || DH == 128) ? 2 : ::relpos::kStages;
  static constexpr uint32_t kHalves = (MODE == 4 || DH == 128) ? 2u : 1u;
  static constexpr uint32_t kQBytes = kHalves * kTileBytes;                         // one query tile
  static constexpr uint32_t kKBytes = kHalves * kTileBytes;                         // one K stage
  // one V stage; DeBERTa appends its keys' two saturated p2c values (2 x 128 fp32)
  static constexpr uint32_t kVBytes = static_cast<uint32_t>(DH / 64) * kTileBytes + (MODE == 2 ? 1024u : 0u);
  static constexpr uint32_t kOffQ = 0;
  static constexpr uint32_t kOffK = kOffQ + 2 * kQBytes;
  static constexpr uint32_t kOffV = kOffK + kStages * kKBytes;
  static constexpr uint32_t kOffBar = kOffV + kStages * kVBytes;
  static constexpr uint32_t kOffAux = kOffBar + 512;
};
constexpr uint32_t kCombBytes = 2 * 128 * 8;  // split items: (m, l) of every row, per tile
// TMEM columns: S of query tile x at x * 128, O at 256 + x * d, P (bf16
// pairs) at 384 + x * 64; at d = 128, P takes the first 64 columns of its
// tile's S (read out by then), whose next S product then waits for the P.V
// that reads it.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;
constexpr uint32_t kTmemO = 256;
constexpr uint32_t kTmemP = 384;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

enum : uint32_t {
  kBarQFull = 0,
  kBarQEmpty = 1,
  kBarKFull = 2,
  kBarVFull = kBarKFull + kStages,
  kBarKEmpty = kBarVFull + kStages,   // K stage read by every S product of its tile
  kBarVEmpty = kBarKEmpty + kStages,  // V stage read by every P.V product of its tile
  kBarSFull = kBarVEmpty + kStages,   // + tile (2)
  kBarSFree = kBarSFull + 2,  // + tile: the softmax has read S out of TMEM
  kBarPFull = kBarSFree + 2,
  kBarODone = kBarPFull + 2,
  kBarOFree = kBarODone + 2,
  kBarTab = kBarOFree + 2,
  kBarComb = kBarTab + 2,  // both softmax warpgroups have published a split item's partial state
  kBarStag = kBarComb + 1,  // + item parity: warpgroup a is past the maximum of its first tile
  kBarFinal = kBarStag + 2,
  kBarQa = kBarFinal + 1,   // + tile, Shaw: q . a_K of the item's rows in TMEM
  kBarWb = kBarQa + 2,      // + tile, Shaw: the value-side bins staged as an operand (128 arrivals)
  kBarOv = kBarWb + 2,      // + tile, Shaw: O += bins . a_V done
  kBarTbl = kBarOv + 2,     // Shaw: the a_K / a_V operand tiles are written (256 arrivals)
  kNumBars = kBarTbl + 1,
};
constexpr uint32_t kOffTmemSlot = 320;
constexpr uint32_t kOffAbort = 324;
static_assert(kNumBars * 8 <= kOffTmemSlot, "barrier block overflow");

constexpr uint32_t kIdescQK = idesc_bf16_f32(kBM, kBN, 0, 0);       // Q, K both K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, kHeadDim, 0, 1);  // P (TMEM), V MN-major
constexpr uint32_t kIdescQa = idesc_bf16_f32(kBM, 64, 0, 0);        // Shaw: Q . a_K^T (64 table rows)

RP_DEVI void record_error(int* status) {
  if (status) atomicCAS(status, 0, -4);
}

// One work item. A pair item holds query rows [i0, i0 + 256) of head bh as
// tiles a (rows from i0) and b (rows from i0 + 128); both visit the same key
// tiles, which stream through shared memory once. A split item holds a single
// 128-row query tile whose key tiles are divided between the two softmax
// warpgroups: a takes [0, na), b takes [na, n), and their partial softmax
// states are merged when both are done. The last items of the list (the
// shortest pairs) are split when that shortens the grid's final pass.
struct Item {
  int bh, h;
  int row0[2];       // first query row of tile a / b
  int lo[2], hi[2];  // key tiles [lo, hi) of tile a / b (none when lo == hi)
  int ns;            // key tiles streamed through shared memory for the item
  bool split;
};

// Valid query rows and keys of (batch, head) bh: the batch element's length
// in a right-padded batch (PAD: the launch variant that takes lengths),
// otherwise no limit.
// Predicated shared-memory store without a branch: a lane whose predicate
// is off does not store.
RP_DEVI void st_shared_f32_if(uint32_t addr, float v, int pred) {
  asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t@q st.shared.f32 [%0], %1;\n\t}" ::"r"(addr), "f"(v),
               "r"(pred)
               : "memory");
}

// 8 consecutive 32-bit TMEM columns of this thread's lane, waited for.
RP_DEVI void tmem_ld8_sync(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
      : "r"(taddr)
      : "memory");
}

template <bool PAD>
RP_DEVI int seq_len(const FwdParams& p, int bh) {
  if constexpr (!PAD) return 0x7fffffff;
  const int n = __ldg(p.lengths + bh / p.H);
  return n < 0 ? 0 : n;
}

// Key tiles [0, n) one 128-row query tile starting at row r0 visits, for a
// sequence of nlen valid rows and keys (a padded batch element; rows from
// nlen on give zero rows). With explicit key positions (POS) a key's index
// says nothing about its position: every tile is visited.
template <bool PAD, bool POS = false>
RP_DEVI int tile_keys(const FwdParams& p, int r0, int nlen) {
  const int lq = PAD ? min(p.Lq, nlen) : p.Lq;
  const int lk = PAD ? min(p.Lk, nlen) : p.Lk;
  if (r0 >= lq || (PAD && lk <= 0)) return 0;
  int last_key = lk - 1;
  if (p.causal && !POS) last_key = min(last_key, min(r0 + kBM - 1, lq - 1) + p.q_offset);
  return last_key / kBN + 1;
}

// SPLIT: the launch has split items (p.nsplit > 0); without, the split paths
// compile away. PAD: a right-padded batch (p.lengths).
template <bool SPLIT, bool PAD, bool POS = false>
RP_DEVI Item make_item(const FwdParams& p, int w) {
  Item it;
  const int BH = p.B * p.H;
  const int whole = p.npairs * BH - (SPLIT ? p.nsplit : 0);  // pair items kept whole
  int wp = w, xs = -1;
  if (SPLIT && w >= whole) {
    wp = whole + ((w - whole) >> 1);
    xs = (w - whole) & 1;
  }
  const int pair = p.npairs - 1 - wp / BH;  // longest (causal) pairs first
  it.bh = wp % BH;
  it.h = it.bh % p.H;
  const int i0 = pair * 2 * kBM;
  const int nlen = seq_len<PAD>(p, it.bh);
  if (xs < 0) {
    it.split = false;
#pragma unroll
    for (int x = 0; x < 2; ++x) {
      it.row0[x] = i0 + x * kBM;
      it.lo[x] = 0;
      it.hi[x] = tile_keys<PAD, POS>(p, it.row0[x], nlen);
    }
    it.ns = max(it.hi[0], it.hi[1]);
  } else {
    it.split = true;
    const int r0 = i0 + xs * kBM;
    const int n = tile_keys<PAD, POS>(p, r0, nlen);
    const int na = (n + 1) >> 1;
    it.row0[0] = it.row0[1] = r0;
    it.lo[0] = 0;
    it.hi[0] = na;
    it.lo[1] = na;
    it.hi[1] = n;
    it.ns = n;
  }
  return it;
}

// Stream position s of an item: the key tile loaded there, and whether query
// tile x uses it. A split item alternates a's and b's key tiles.
RP_DEVI int stream_key(const Item& it, int s) {
  return it.split ? ((s & 1) ? it.lo[1] + (s >> 1) : (s >> 1)) : s;
}
RP_DEVI bool stream_uses(const Item& it, int x, int s) {
  return it.split ? (s & 1) == x : s < (x ? it.hi[1] : it.hi[0]);
}
// Field x of an item, selected without indexing (keeps the item in registers).
RP_DEVI int sel(const int (&v)[2], int x) { return x ? v[1] : v[0]; }

// The item a CTA takes in its r-th pass over the grid (pass r covers items
// r * grid ... r * grid + grid - 1): items are ordered longest first. With
// causal masking the CTAs sweep them in alternating directions (pass 0 left
// to right, pass 1 right to left, ...) so that long and short items pair
// up. Otherwise every item is equally long and every pass goes left to
// right: CTAs are dispatched in index order, so the lowest indices start
// first and those take the extra items of a final partial pass.
RP_DEVI int item_at(int r, bool snake) {
  const int g = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
  return r * g + ((snake && (r & 1)) ? g - 1 - c : c);
}

// Head of the first item from pass r on in which query tile x has key tiles,
// or -1.
template <bool SPLIT, bool PAD, bool POS = false>
RP_DEVI int next_head(const FwdParams& p, int x, int r, int nitems) {
  for (int w = item_at(r, p.causal); w < nitems; w = item_at(++r, p.causal)) {
    const Item it = make_item<SPLIT, PAD, POS>(p, w);
    if (sel(it.hi, x) > sel(it.lo, x)) return it.h;
  }
  return -1;
}

// T5 per-WG bias-by-offset table: 4 copies shifted by one entry each, so any
// run of 128 consecutive offsets starts 16-byte aligned in one of them. A lane
// reads copy (s & 3) for its window start s, and the lanes of a quarter-warp
// hold 8 consecutive starts. Copy k is placed off[k] 16-byte chunks into its
// 128-byte-aligned slot so that those 8 reads land on 8 distinct bank groups:
// with r = (lowest start of the quarter) & 3, the rank q = (k - r) & 3 takes
// chunk offset 2q, minus one for the copies whose windows begin one chunk
// further on (k < r).
// When the four copies do not fit shared memory (long saturation distance),
// the table is kept as one copy read one entry per load ("compact").
struct T5Tab {
  float* base;  // [2 buffers][ncopy copies][stride]
  int len4;     // entries per copy
  int stride;   // floats per copy slot (multiple of 32, >= len4 + 28)
  int ncopy;    // 4, or 1 (compact)
  int r;
  RP_DEVI float* copy(int buf, int k) const {
    const int q = (k - r) & 3;
    const int off = (2 * q - (k < r ? 1 : 0)) & 7;
    return base + (buf * ncopy + k) * stride + 4 * off;
  }
};

RP_DEVI int t5_copy_stride(int len4) { return (len4 + 28 + 31) & ~31; }

// Shaw's tables after kOffAux (which sits 512 bytes past a 1024-byte
// boundary): the a_K and a_V tiles (64 rows x 128 bytes, 128-byte swizzle,
// rows past 2k zero; the B operands of the q . a_K product and of the value
// product), then per warpgroup a region holding its rows' q . a_K values
// during an item and, at the item's end, its rows' value-side bins as the
// bf16 A operand of the value product (a 16 KB tile), then the bins
// themselves (fp32, per row).
struct ShawAux {
  uint32_t tK, tV, qa0, rq, wbin, end;
};
__host__ __device__ inline ShawAux shaw_aux(int row_stride) {
  ShawAux a;
  a.tK = 512u;
  a.tV = a.tK + 8192u;
  a.qa0 = a.tV + 8192u;
  uint32_t rq = 128u * static_cast<uint32_t>(row_stride) * 4u;
  if (rq < 16384u) rq = 16384u;
  a.rq = (rq + 1023u) & ~1023u;
  a.wbin = a.qa0 + 2u * a.rq;
  a.end = a.wbin + 256u * static_cast<uint32_t>(row_stride) * 4u;
  return a;
}

// Bytes of the mode's relative-term tables after kOffAux (16-byte multiple);
// the split-item (m, l) exchange follows them.
__host__ __device__ inline uint32_t fwd_aux_bytes(int mode, const FwdParams& p) {
  uint32_t aux = 0;
  if (mode == 0) {
    const uint32_t bkt_bytes = (static_cast<uint32_t>(p.t5_tab_len4) + 4u + 127u) & ~127u;
    const uint32_t stride = (static_cast<uint32_t>(p.t5_tab_len4) + 28u + 31u) & ~31u;
    const uint32_t ncopy = p.t5_compact ? 1u : 4u;
    aux = bkt_bytes + 2u * 2u * ncopy * stride * 4u + 2u * 128u * 4u;
    aux = (aux + 15u) & ~15u;
    if (p.key_pos) aux += 8u * 128u * 4u;  // each softmax warp's key positions of a tile
  } else if (mode == 1) {
    aux = shaw_aux(p.row_stride).end;
  }
  return (aux + 15u) & ~15u;
}

// VAR 0: pair items only; 1: with split items (p.nsplit > 0); 2: pair items
// with the two softmax warpgroups staggered (p.stagger); 3: pair items of a
// right-padded batch (p.lengths); 4: T5 pair items over keys at explicit
// positions (p.key_pos).
// Loads one query tile (both halves for Transformer-XL and d = 128) on
// barrier `bar`.
template <int MD, bool ELECT>
RP_DEVI void load_q_tile(uint32_t dst, const CUtensorMap* tmQ, uint32_t bar, int row0, int bh) {
#pragma unroll
  for (uint32_t h = 0; h < Smem<MD>::kHalves; ++h) {
    if constexpr (ELECT)
      tma_load_3d_elect(dst + h * kTileBytes, tmQ, bar, static_cast<int>(h) * kHeadDim, row0, bh);
    else
      tma_load_3d(dst + h * kTileBytes, tmQ, bar, static_cast<int>(h) * kHeadDim, row0, bh);
  }
}
// Loads one K stage: the key tile and, for Transformer-XL, the keys'
// sinusoid rows (one [Lk, 64] table for every head) as the second half; at
// d = 128 the key rows' two halves.
template <int MD, bool ELECT>
RP_DEVI void load_k_stage(uint32_t dst, const CUtensorMap* tmK, const CUtensorMap* tmS, uint32_t bar,
                          int key0, int bh) {
  constexpr int MODE = md_mode(MD);
  if constexpr (ELECT) {
    tma_load_3d_elect(dst, tmK, bar, 0, key0, bh);
    if constexpr (MODE == 4) tma_load_3d_elect(dst + kTileBytes, tmS, bar, 0, key0, 0);
    if constexpr (md_dim(MD) == 128) tma_load_3d_elect(dst + kTileBytes, tmK, bar, 64, key0, bh);
  } else {
    tma_load_3d(dst, tmK, bar, 0, key0, bh);
    if constexpr (MODE == 4) tma_load_3d(dst + kTileBytes, tmS, bar, 0, key0, 0);
    if constexpr (md_dim(MD) == 128) tma_load_3d(dst + kTileBytes, tmK, bar, 64, key0, bh);
  }
}
// Bulk copy of `bytes` contiguous global bytes into shared memory on barrier
// `bar` (both addresses 16-byte aligned, bytes a multiple of 16); the _elect
// form is issued by one elected lane of a converged warp.
RP_DEVI void bulk_load_1d(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
RP_DEVI void bulk_load_1d_elect(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n\t}" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// Loads one V stage (both 64-column halves at d = 128; DeBERTa also the
// keys' saturated p2c values, far behind then far ahead, 512 bytes each).
template <int MD, bool ELECT>
RP_DEVI void load_v_stage(uint32_t dst, const CUtensorMap* tmV, uint32_t bar, int key0, int bh,
                          const FwdParams& p) {
#pragma unroll
  for (int h = 0; h < md_dim(MD) / 64; ++h) {
    if constexpr (ELECT)
      tma_load_3d_elect(dst + h * kTileBytes, tmV, bar, 64 * h, key0, bh);
    else
      tma_load_3d(dst + h * kTileBytes, tmV, bar, 64 * h, key0, bh);
  }
  if constexpr (md_mode(MD) == 2) {
    const float* e = p.p2c_ends + static_cast<size_t>(bh) * 2 * p.ends_pitch + key0;
    if constexpr (ELECT) {
      bulk_load_1d_elect(dst + kTileBytes, e, 512u, bar);
      bulk_load_1d_elect(dst + kTileBytes + 512u, e + p.ends_pitch, 512u, bar);
    } else {
      bulk_load_1d(dst + kTileBytes, e, 512u, bar);
      bulk_load_1d(dst + kTileBytes + 512u, e + p.ends_pitch, 512u, bar);
    }
  }
}

template <int MD, bool OUT_F32, int VAR>
__global__ void __launch_bounds__(kThreads, 1)
    relpos_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmS,
                      const FwdParams p) {
  constexpr int MODE = md_mode(MD);  // 0 T5, 1 Shaw, 2 DeBERTa, 3 ALiBi, 4 Transformer-XL
  constexpr int DH = md_dim(MD);     // head dimension
  constexpr bool SPLIT = VAR == 1;
  constexpr bool STAG = VAR == 2;
  constexpr bool PAD = VAR == 3;
  constexpr bool POS = VAR == 4;  // T5 with explicit key positions (p.key_pos)
  using L = Smem<MD>;
  constexpr uint32_t kOffQ = L::kOffQ, kOffK = L::kOffK, kOffV = L::kOffV, kOffBar = L::kOffBar,
                     kOffAux = L::kOffAux;
  constexpr int kRing = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_addr);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nitems = p.B * p.H * p.npairs + p.nsplit;

  auto bar = [&](uint32_t i) { return sbase + kOffBar + i * 8; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + kOffAbort);

  // ---------------------------------------------------------------- setup
  // Nothing here loads from or writes to global memory (only L2 prefetches of
  // the first tiles), so a launch that follows in the stream may run it
  // early. Each role waits for the previous kernel (griddep_wait) just before
  // its own first global access: the producers before their first load, the
  // softmax warpgroups before their first table read; the MMA issuers touch
  // global memory only to report an error.
  griddep_launch_dependents();
  // a padded batch's lengths are read by every role's item walk, the setup's
  // included: wait for the previous kernel before anything else
  if constexpr (PAD) griddep_wait();
  uint8_t* aux = smem + kOffAux;
  uint8_t* bkt = aux;  // T5: head-independent bucket of each table offset
  const int nrel = 2 * p.kclip + 1;
  const ShawAux shaw = shaw_aux(p.row_stride);
  if constexpr (MODE == 0) {
    for (int x = threadIdx.x; x < p.t5_tab_len4 + 4; x += kThreads) {
      const int xc = min(x, p.t5_tab_len - 1);
      bkt[x] = static_cast<uint8_t>(t5_bucket_dev(xc - p.t5_tab_off, p.t5));
    }
  }
  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < kNumBars; ++i) {
      uint32_t cnt = 1;
      if (i == kBarPFull || i == kBarPFull + 1 || i == kBarTab || i == kBarTab + 1 ||
          i == kBarSFree || i == kBarSFree + 1 || i == kBarStag || i == kBarStag + 1)
        cnt = 128;  // every thread of a softmax warpgroup
      if (i == kBarOFree || i == kBarOFree + 1 || i == kBarComb)
        cnt = 256;  // both softmax warpgroups (or one, arriving twice)
      if (i == kBarWb || i == kBarWb + 1) cnt = 128;
      if (i == kBarTbl) cnt = 256;
      if (i == kBarQEmpty || i == kBarFinal || (i >= kBarKEmpty && i < kBarVEmpty + kStages))
        cnt = 2;    // both MMA issuers
      mbar_init(bar(i), cnt);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + kOffBar + kOffTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  // This CTA's first item: its Q tile(s) and first K / V ring stages are
  // warmed in L2 while the previous kernel finishes (L2 is coherent, so the
  // loads after the wait see its writes), then loaded by this thread as soon
  // as the inputs may be read; the producer loops start after them.
  const bool first_loads = threadIdx.x == 0 && static_cast<int>(blockIdx.x) < nitems;
  Item it0{};
  bool two0 = false;
  int nk0 = 0;
  if (first_loads) {
    it0 = make_item<SPLIT, PAD, POS>(p, item_at(0, p.causal));
    two0 = !it0.split && it0.hi[1] > 0;
    nk0 = it0.ns < kRing ? it0.ns : kRing;
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    if constexpr (MODE == 4) tma_prefetch_desc(&tmS);
    for (uint32_t hf = 0; hf < L::kHalves; ++hf) {
      tma_prefetch_l2_3d(&tmQ, hf * kHeadDim, it0.row0[0], it0.bh);
      if (two0) tma_prefetch_l2_3d(&tmQ, hf * kHeadDim, it0.row0[1], it0.bh);
    }
    for (int s = 0; s < nk0; ++s) {
      tma_prefetch_l2_3d(&tmK, 0, stream_key(it0, s) * kBN, it0.bh);
      tma_prefetch_l2_3d(&tmV, 0, stream_key(it0, s) * kBN, it0.bh);
    }
    if constexpr (MODE == 0) {
      // the bias rows, read by the softmax warpgroups first thing
      const int lines = min((p.t5_nb * p.H * 4 + 127) / 128, 64);
      for (int l = 0; l < lines; ++l) prefetch_l2(reinterpret_cast<const char*>(p.bias) + l * 128);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffBar + kOffTmemSlot);

  if (warp < 4) {
    // register split (4 x 32 x dec + 8 x 32 x inc <= 384 x 168): T5 needs
    // fewer in the softmax and gives its issuers room (not with explicit key
    // positions, whose per-element path needs the softmax's share)
    if constexpr (MODE == 0 && !POS) {
      setmaxnreg_dec<88>();
    } else {
      setmaxnreg_dec<72>();
    }
    if (warp == 0 || warp == 2) {
      // ------------------------------------------------------------ producers
      // warp 0: each item's Q tiles and the K ring; warp 2: the V ring
      const bool kq = warp == 0;
      griddep_wait();
      if (first_loads) {
        mbar_arrive_expect_tx(bar(kBarQFull), (two0 ? 2u : 1u) * L::kQBytes);
        load_q_tile<MD, false>(sbase + kOffQ, &tmQ, bar(kBarQFull), it0.row0[0], it0.bh);
        if (two0) load_q_tile<MD, false>(sbase + kOffQ + L::kQBytes, &tmQ, bar(kBarQFull), it0.row0[1], it0.bh);
        for (int s = 0; s < nk0; ++s) {
          const int key0 = stream_key(it0, s) * kBN;
          mbar_arrive_expect_tx(bar(kBarKFull + s), L::kKBytes);
          load_k_stage<MD, false>(sbase + kOffK + s * L::kKBytes, &tmK, &tmS, bar(kBarKFull + s), key0, it0.bh);
          mbar_arrive_expect_tx(bar(kBarVFull + s), L::kVBytes);
          load_v_stage<MD, false>(sbase + kOffV + s * L::kVBytes, &tmV, bar(kBarVFull + s), key0, it0.bh, p);
        }
      }
      const uint32_t full0 = kq ? kBarKFull : kBarVFull;
      const uint32_t empty0 = kq ? kBarKEmpty : kBarVEmpty;
      const uint32_t ring = kq ? kOffK : kOffV;
      const uint32_t stage_bytes = kq ? L::kKBytes : L::kVBytes;
      bool ok = true;
      uint32_t it_cnt = 0;
      int item_cnt = 0;
      for (int rr = 0, w = item_at(0, p.causal); ok && w < nitems; w = item_at(++rr, p.causal), ++item_cnt) {
        const Item it = make_item<SPLIT, PAD, POS>(p, w);
        // the first item's Q and first ring stages were loaded in the setup
        const int pre = item_cnt == 0 ? min(it.ns, kRing) : 0;
        if (kq && item_cnt > 0) {
          ok = mbar_wait_warp(bar(kBarQEmpty), (item_cnt - 1) & 1);
          if (!ok) break;
          // a split item's single query tile goes to the Q_a buffer
          const bool two = !it.split && it.hi[1] > 0;
          mbar_arrive_expect_tx_elect(bar(kBarQFull), (two ? 2u : 1u) * L::kQBytes);
          load_q_tile<MD, true>(sbase + kOffQ, &tmQ, bar(kBarQFull), it.row0[0], it.bh);
          if (two) load_q_tile<MD, true>(sbase + kOffQ + L::kQBytes, &tmQ, bar(kBarQFull), it.row0[1], it.bh);
        }
        for (int j = 0; j < it.ns; ++j, ++it_cnt) {
          if (j < pre) continue;
          const uint32_t st = it_cnt % kRing;
          if (it_cnt >= kRing) {
            ok = mbar_wait_warp(bar(empty0 + st), ((it_cnt / kRing) - 1) & 1);
            if (!ok) break;
          }
          mbar_arrive_expect_tx_elect(bar(full0 + st), stage_bytes);
          if (kq)
            load_k_stage<MD, true>(sbase + ring + st * stage_bytes, &tmK, &tmS, bar(full0 + st),
                                     stream_key(it, j) * kBN, it.bh);
          else
            load_v_stage<MD, true>(sbase + ring + st * stage_bytes, &tmV, bar(full0 + st),
                                   stream_key(it, j) * kBN, it.bh, p);
        }
      }
      if (!ok && lane == 0) {
        record_error(p.status);
        *abort_flag = 1;
      }
      // never leave with copies in flight: wait (bounded) for the last loads
      const uint32_t first = it_cnt > kRing ? it_cnt - kRing : 0;
      for (uint32_t k = first; k < it_cnt; ++k)
        mbar_wait_warp(bar(full0 + k % kRing), (k / kRing) & 1, 100000000ull);
      if (kq && item_cnt > 0) mbar_wait_warp(bar(kBarQFull), (item_cnt - 1) & 1, 100000000ull);
    } else if (warp == 1 || warp == 3) {
      // ------------------------------------------------------------ MMA issuers
      // Warp 1 issues the products of query tile a, warp 3 those of tile b, so
      // each reacts only to its own softmax warpgroup. For its key tiles in
      // stream order: S = Q K^T of the next tile as soon as the softmax has
      // read the previous S, then O += P V of the current tile as soon as P is
      // in TMEM. Stream positions of the other tile only are released without
      // use. K / V stages and the Q buffers are freed once both issuers are
      // done with them (barriers counting two arrivals).
      const uint32_t x = warp == 1 ? 0u : 1u;
      bool ok = true;
      uint32_t kv_it = 0;  // ring position of the item's first key tile
      uint32_t sis = 0;    // S products issued
      uint32_t pvc = 0;    // P.V products issued
      uint32_t ocnt = 0;   // items whose O accumulator this issuer used
      int item_cnt = 0;
      // descriptors at K-step 0; later K-steps add the step's byte offset / 16
      const uint64_t dq_a = smem_desc_sw128(sbase + kOffQ, 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(sbase + kOffK, 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(sbase + kOffV, 8192, 1024);
      constexpr uint64_t kStageStep = kTileBytes >> 4;  // one 64-column tile
      constexpr uint64_t kQStep = L::kQBytes >> 4, kKStep = L::kKBytes >> 4, kVStep = L::kVBytes >> 4;
      const uint32_t s_col = tmem + kTmemS + x * kBN;
      const uint32_t o_col = tmem + kTmemO + x * DH;
      const uint32_t p_col = DH == 128 ? s_col : tmem + kTmemP + x * 64;
      for (int rr = 0, w = item_at(0, p.causal); ok && w < nitems; w = item_at(++rr, p.causal), ++item_cnt) {
        const Item it = make_item<SPLIT, PAD, POS>(p, w);
        const int mine = sel(it.hi, x) - sel(it.lo, x);
        const uint64_t dq = dq_a + ((it.split ? 0u : x) * kQStep);
        ok = mbar_wait_warp(bar(kBarQFull), item_cnt & 1);
        if (!ok) break;
        if (mine == 0 && lane == 0) mbar_arrive(bar(kBarQEmpty));
        int kpos = 0, vpos = 0;  // next stream positions of the K and V rings
        // Release the K (or V) stages of the other tile's positions up to this
        // tile's next one; returns that position, or it.ns when none is left.
        auto advance = [&](int& pos, uint32_t full0, uint32_t empty0) -> int {
          while (pos < it.ns && !stream_uses(it, x, pos)) {
            const uint32_t r = kv_it + pos;
            ok = mbar_wait_warp(bar(full0 + r % kRing), (r / kRing) & 1);
            if (!ok) return it.ns;
            if (lane == 0) mbar_arrive(bar(empty0 + r % kRing));
            ++pos;
          }
          return pos;
        };
        // S of this tile's i-th key tile (at the K cursor)
        auto issue_s = [&](int i) -> bool {
          const int pos = advance(kpos, kBarKFull, kBarKEmpty);
          if (!ok) return false;
          const uint32_t r = kv_it + pos;
          const uint32_t st = r % kRing;
          if (!mbar_wait_warp(bar(kBarKFull + st), (r / kRing) & 1)) return false;
          if (sis > 0 && !mbar_wait_warp(bar(kBarSFree + x), (sis - 1) & 1)) return false;
          // d = 128: P lives in this S's columns; the P.V that reads it first
          if (DH == 128 && pvc > 0 && !mbar_wait_warp(bar(kBarODone + x), (pvc - 1) & 1)) return false;
          tc_fence_after();
          const uint64_t dk = dk0 + st * kKStep;
          // K-steps of 16: 4 per 64-column half (Transformer-XL: content, then position)
#pragma unroll
          for (int kk = 0; kk < static_cast<int>(L::kHalves) * (kHeadDim / 16); ++kk) {
            const uint64_t off = (kk >> 2) * kStageStep + 2 * (kk & 3);
            umma_bf16_ss_elect(s_col, dq + off, dk + off, kIdescQK, kk > 0 ? 1u : 0u);
          }
          tc_commit_elect(bar(kBarSFull + x));
          tc_commit_elect(bar(kBarKEmpty + st));
          if (i == mine - 1) tc_commit_elect(bar(kBarQEmpty));
          ++sis;
          ++kpos;
          return true;
        };
        if constexpr (MODE == 1) {
          // Shaw: q . a_K[r] of every row of the item's tile (Q . a_K^T, 64
          // table rows, the rows past 2k zero) into this tile's O accumulator,
          // which the previous item's epilogue has read; the softmax reads
          // it back before its first P.V
          if (mine > 0) {
            if (ocnt == 0) ok = mbar_wait_warp(bar(kBarTbl), 0);
            if (ok && ocnt > 0) ok = mbar_wait_warp(bar(kBarOFree + x), (ocnt - 1) & 1);
            if (!ok) break;
            tc_fence_after();
            const uint64_t dta = smem_desc_sw128(sbase + kOffAux + shaw.tK, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < kHeadDim / 16; ++kk)
              umma_bf16_ss_elect(o_col, dq + 2 * kk, dta + 2 * kk, kIdescQa, kk > 0 ? 1u : 0u);
            tc_commit_elect(bar(kBarQa + x));
          }
        }
        if (mine > 0) ok = issue_s(0);
        for (int i = 0; ok && i < mine; ++i) {
          // look ahead: the next key tile's scores (after the last one, free
          // the other tile's remaining K stages at once); at d = 128 after
          // this tile's P.V, which reads the columns the next S writes
          if (DH == 64) {
            if (i + 1 < mine) {
              ok = issue_s(i + 1);
              if (!ok) break;
            } else {
              advance(kpos, kBarKFull, kBarKEmpty);
              if (!ok) break;
            }
          }
          // this key tile's P.V
          const int pos = advance(vpos, kBarVFull, kBarVEmpty);
          if (!ok) break;
          const uint32_t r = kv_it + pos;
          const uint32_t st = r % kRing;
          ok = mbar_wait_warp(bar(kBarPFull + x), pvc & 1);
          if (MODE != 1 && ok && i == 0 && ocnt > 0) ok = mbar_wait_warp(bar(kBarOFree + x), (ocnt - 1) & 1);
          if (ok) ok = mbar_wait_warp(bar(kBarVFull + st), (r / kRing) & 1);
          tc_fence_after();
          if (!ok) break;
          const uint64_t dv = dv0 + st * kVStep;
#pragma unroll
          for (int hc = 0; hc < DH / 64; ++hc)  // 64 output columns per V half
#pragma unroll
            for (int kk = 0; kk < kBN / 16; ++kk)
              umma_bf16_ts_elect(o_col + 64 * hc, p_col + kk * 8, dv + hc * kStageStep + 128 * kk, kIdescPV,
                                 (i > 0 || kk > 0) ? 1u : 0u);
          tc_commit_elect(bar(kBarODone + x));
          tc_commit_elect(bar(kBarVEmpty + st));
          ++pvc;
          ++vpos;
          if (DH == 128) {
            if (i + 1 < mine) {
              ok = issue_s(i + 1);
              if (!ok) break;
            } else {
              advance(kpos, kBarKFull, kBarKEmpty);
              if (!ok) break;
            }
          }
        }
        if constexpr (MODE == 1) {
          // Shaw: O += bins . a_V once the softmax has staged its rows' bins
          if (ok && mine > 0) {
            ok = mbar_wait_warp(bar(kBarWb + x), ocnt & 1);
            if (!ok) break;
            tc_fence_after();
            const uint64_t dwb = smem_desc_sw128(sbase + kOffAux + shaw.qa0 + x * shaw.rq, 16, 1024);
            const uint64_t dtv = smem_desc_sw128(sbase + kOffAux + shaw.tV, 8192, 1024);
#pragma unroll
            for (int kk = 0; kk < 64 / 16; ++kk)
              umma_bf16_ss_elect(o_col, dwb + 2 * kk, dtv + 128 * kk, kIdescPV, 1u);
            tc_commit_elect(bar(kBarOv + x));
          }
        }
        // The other tile's remaining positions, K and V stage of each position
        // together: releasing every K stage first could wait for a K load that
        // needs a V stage this warp has not released yet (through the other
        // issuer, whose P.V waits for that V stage).
        for (int pos = min(kpos, vpos); ok && pos < it.ns; ++pos) {
          const uint32_t r = kv_it + pos;
          if (pos >= kpos) {
            ok = mbar_wait_warp(bar(kBarKFull + r % kRing), (r / kRing) & 1);
            if (ok && lane == 0) mbar_arrive(bar(kBarKEmpty + r % kRing));
          }
          if (ok && pos >= vpos) {
            ok = mbar_wait_warp(bar(kBarVFull + r % kRing), (r / kRing) & 1);
            if (ok && lane == 0) mbar_arrive(bar(kBarVEmpty + r % kRing));
          }
        }
        kv_it += it.ns;
        if (mine > 0) ++ocnt;
      }
      if (!ok && lane == 0) {
        griddep_wait();
        record_error(p.status);
        *abort_flag = 1;
      }
      tc_commit_elect(bar(kBarFinal));
      mbar_wait_warp(bar(kBarFinal), 0, 100000000ull);
    }
  } else {
    if constexpr (MODE == 0 && !POS) {
      setmaxnreg_inc<200>();
    } else {
      setmaxnreg_inc<216>();
    }
    // -------------------------------------------------------------- softmax
    const int x = (warp - 4) >> 2;                  // query tile a (0) or b (1)
    const int t = ((warp & 3) << 5) | lane;          // row == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_base + kTmemS + x * kBN;
    const uint32_t tO = tmem + lane_base + kTmemO + x * DH;
    const uint32_t tP = DH == 128 ? tS : tmem + lane_base + kTmemP + x * 64;
    const float sl2 = p.scale_log2;
    const float kNegInf = -INFINITY;
    bool err = false;
    if constexpr (MODE == 1) {
      // the relative key / value tables as tensor-core operands: row r holds
      // a_K[r] (a_V[r]), 16-byte chunks swizzled by the row, rows past 2k zero
      griddep_wait();
      const uint4* srcK = reinterpret_cast<const uint4*>(p.aK);
      const uint4* srcV = reinterpret_cast<const uint4*>(p.aV);
      for (int i = static_cast<int>(threadIdx.x) - 128; i < 64 * 8; i += 256) {
        const int r = i >> 3, c = i & 7;
        const uint32_t off = static_cast<uint32_t>(r) * 128u + (static_cast<uint32_t>(c ^ (r & 7)) << 4);
        const bool in = r < nrel;
        *reinterpret_cast<uint4*>(aux + shaw.tK + off) = in ? __ldg(srcK + r * 8 + c) : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4*>(aux + shaw.tV + off) = in ? __ldg(srcV + r * 8 + c) : make_uint4(0u, 0u, 0u, 0u);
      }
      // visible to the tensor core, then to the issuers (their first
      // q . a_K product waits for this)
      fence_async_smem();
      mbar_arrive(bar(kBarTbl));
    }

    T5Tab tab{};
    float* hbias = nullptr;  // T5: this head's bias per bucket (log2 units)
    float hb_next = 0.f;     // T5: thread t < num_buckets holds entry t of the next table's row
    float* qa = nullptr;    // Shaw: q . a_K[r] of this row (log2 units)
    float* wbin = nullptr;  // Shaw: probability mass per clipped offset of this row
    uint8_t* wb_tile = nullptr;  // Shaw: this warpgroup's bins operand (over its q . a_K rows)
    if constexpr (MODE == 0) {
      tab.len4 = p.t5_tab_len4;
      tab.stride = t5_copy_stride(p.t5_tab_len4);
      // every window start is j0 - (i0 + 32 w + lane + q_offset) + tab_off with
      // j0, i0, 32 w multiples of 4: the lowest start of a quarter-warp is
      // (tab_off - q_offset - 7) mod 4
      tab.r = (((p.t5_tab_off - p.q_offset - 7) % 4) + 4) % 4;
      const uint32_t bkt_bytes = (static_cast<uint32_t>(p.t5_tab_len4) + 4u + 127u) & ~127u;
      tab.ncopy = p.t5_compact ? 1 : 4;
      tab.base = reinterpret_cast<float*>(aux + bkt_bytes) + x * 2 * tab.ncopy * tab.stride;
      hbias = reinterpret_cast<float*>(aux + bkt_bytes) + 2 * 2 * tab.ncopy * tab.stride + x * 128;
    } else if constexpr (MODE == 1) {
      // rows p.row_stride floats apart: with 2k + 2 (even), the lanes of a
      // near tile, which read offsets r0 - t + c of their rows, hit distinct
      // banks (with 2k + 1 they are 2k words apart: one bank)
      wb_tile = aux + shaw.qa0 + x * shaw.rq;
      qa = reinterpret_cast<float*>(wb_tile) + t * p.row_stride;
      wbin = reinterpret_cast<float*>(aux + shaw.wbin) + (x * 128 + t) * p.row_stride;
    }
    const int kc = p.kclip;

    // T5: fill table buffer b from the bias row in hb_next. The Tab barrier
    // completes twice per table: once the row is staged in shared memory, and
    // once every entry is written (awaited when the item starts).
    auto t5_build = [&](int b) -> bool {
      if (t < p.t5_nb) hbias[t] = hb_next * kLog2e;
      mbar_arrive(bar(kBarTab + x));
      if (!mbar_wait(bar(kBarTab + x), 0)) return false;
      for (int y = 4 * t; y < tab.len4; y += 4 * 128) {
        const uint32_t w0 = *reinterpret_cast<const uint32_t*>(bkt + y);
        const uint32_t w1 = *reinterpret_cast<const uint32_t*>(bkt + y + 4);
        float v[7];
#pragma unroll
        for (int e = 0; e < 4; ++e) v[e] = hbias[(w0 >> (8 * e)) & 0xffu];
#pragma unroll
        for (int e = 0; e < 3; ++e) v[4 + e] = hbias[(w1 >> (8 * e)) & 0xffu];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (k < tab.ncopy)
            *reinterpret_cast<float4*>(tab.copy(b, k) + y) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
      }
      mbar_arrive(bar(kBarTab + x));
      return true;
    };
    if constexpr (MODE == 0) {
      const int h0 = next_head<SPLIT, PAD, POS>(p, x, 0, nitems);
      griddep_wait();
      if (h0 >= 0) {
        if (t < p.t5_nb) hb_next = __ldg(p.bias + t * p.H + h0);
        if (!t5_build(0)) err = true;
      }
    }

    if constexpr (MODE >= 2) griddep_wait();
    uint32_t cnt = 0, ocnt = 0;
    uint32_t ccnt = 0;  // split items merged with the other warpgroup
    // With STAG, warpgroup b starts each item once warpgroup a has its
    // first tile's maximum, so that the two run about half a tile apart and
    // their exponential phases (MUFU) overlap the other's score and maximum
    // phases instead of each other. It pays on long items of mostly far
    // tiles (causal T5, causal Transformer-XL); elsewhere it gains nothing
    // or, on short items, the later start of b costs more.
    // `stag` counts the items in which a has key tiles; the item's turn goes
    // to one of two alternating barriers: a can lead b by at most two items
    // (b has started the last tile of item n - 2 before a's item n has its
    // Q tiles), so two barriers keep the parities apart.
    uint32_t stag = 0;
    uint32_t kv_next = 0;  // DeBERTa: ring position of the next item's first key tile
    float2* ml = reinterpret_cast<float2*>(aux + fwd_aux_bytes(MODE, p));
    for (int rr = 0, w = item_at(0, p.causal); !err && w < nitems; w = item_at(++rr, p.causal)) {
      const Item it = make_item<SPLIT, PAD, POS>(p, w);
      const uint32_t kv_it = kv_next;
      kv_next += static_cast<uint32_t>(it.ns);
      const int lo_x = sel(it.lo, x);
      const int n_kv = sel(it.hi, x) - lo_x;
      const uint32_t stag_it = stag;
      const bool a_has = it.hi[0] > it.lo[0];
      if (x == 0 ? n_kv > 0 : a_has) ++stag;
      const int nlen = seq_len<PAD>(p, it.bh);  // valid rows and keys (padded batches)
      if (n_kv == 0) {
        // a padded batch element's query tile past its length: zero rows
        const int r0 = sel(it.row0, x);
        if (PAD && r0 < p.Lq) {
          const int row = r0 + t;
          if (row < p.Lq) {
            const size_t base = (static_cast<size_t>(it.bh) * p.Lq + row) * DH;
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) + base * (OUT_F32 ? 4 : 2));
#pragma unroll
            for (int c = 0; c < (OUT_F32 ? DH / 4 : DH / 8); ++c) dst[c] = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        continue;
      }
      const int i0 = sel(it.row0, x);
      const int lk_eff = PAD ? min(p.Lk, nlen) : p.Lk;
      const int prow = i0 + t + p.q_offset;  // absolute position of this row
      const int p_lo = i0 + p.q_offset;      // of the tile's first row

      // ---- per-item relative-term setup
      float add_l = 0.f, add_r = 0.f;
      int buf = 0, next_h = -1;
      float alibi_k = 0.f;  // ALiBi: this head's slope in raw-score units (slope / scale)
      if constexpr (MODE == 3) alibi_k = __ldg(p.slopes + it.h) * kLog2e / sl2;
      if constexpr (MODE == 0) {
        // this item's table was filled at the end of the previous item (or in
        // the prologue); fetch the next item's bias row meanwhile
        buf = ocnt & 1;
        next_h = next_head<SPLIT, PAD, POS>(p, x, rr + 1, nitems);
        if (t < p.t5_nb && next_h >= 0) hb_next = __ldg(p.bias + t * p.H + next_h);
        const bool ok = mbar_wait(bar(kBarTab + x), 1);
        err = __any_sync(0xffffffffu, !ok);
        if (err) break;
        add_l = tab.copy(buf, 0)[p.t5_tab_off - p.t5_R];
        add_r = tab.copy(buf, 0)[p.t5_tab_off + p.t5_R];
      } else if constexpr (MODE == 1) {
        // q . a_K[r] for every clipped offset r: the issuer computed Q . a_K^T
        // into this tile's O accumulator before the item's first P.V
        const bool ok = mbar_wait(bar(kBarQa + x), ocnt & 1);
        err = __any_sync(0xffffffffu, !ok);
        if (err) break;
        tc_fence_after();
        uint32_t qr[2][32];
        tmem_ld32(tO, qr[0]);
        tmem_ld32(tO + 32, qr[1]);
        tmem_ld_wait(qr[0]);
        tmem_ld_wait(qr[1]);
        tc_fence_before();
        const float* qv = reinterpret_cast<const float*>(&qr[0][0]);
#pragma unroll
        for (int r = 0; r < 64; ++r) {
          if (r < nrel) {
            qa[r] = qv[r] * sl2;
            wbin[r] = 0.f;
          }
        }
        add_l = qa[0];
        add_r = qa[2 * kc];
      }
      const __nv_bfloat16* band_row = nullptr;  // DeBERTa: this row's band values (log2 units)
      int band_sh = 0;                          // and its shift
      if constexpr (MODE == 2) {
        // rows past Lq read row Lq - 1 (their results are not stored); the
        // shift follows the row's own position, which keeps every window
        // 16-byte aligned
        const int rowc = min(i0 + t, p.Lq - 1);
        band_row = p.band + (static_cast<size_t>(it.bh) * p.Lq + rowc) * p.band_pitch;
        band_sh = (prow - kc) & 7;
        // keys far behind (i - j >= k) take C2P[i][2k - 1]; far ahead, C2P[i][0]
        const float* cc = p.c2p_const + static_cast<size_t>(it.bh) * 2 * p.const_pitch + rowc;
        add_l = cc[0];
        add_r = cc[p.const_pitch];
        // bring this row's windows of the item's band tiles (the pre-pass
        // wrote the array well before: DRAM) into L2 ahead of their loads
        for (int j = 0; j < n_kv; ++j) {
          const int j0 = (lo_x + j) * kBN;
          if (j0 + kBN - 1 - p_lo <= -kc || j0 - (p_lo + kBM - 1) >= kc) continue;  // beyond the band
          const char* wnd = reinterpret_cast<const char*>(band_row + (band_sh + j0 - prow + kc));
          prefetch_l2(wnd);
          prefetch_l2(wnd + 128);
          prefetch_l2(wnd + 255);
        }
      }
      float mass_l = 0.f, mass_r = 0.f;

      float m_run = kNegInf;
      float l_run = 0.f;
      if (STAG && x == 1 && a_has) {
        const bool ok = mbar_wait(bar(kBarStag + (stag_it & 1)), (stag_it >> 1) & 1);
        err = __any_sync(0xffffffffu, !ok);
        if (err) break;
      }
      for (int j = 0; j < n_kv; ++j, ++cnt) {
        const int j0 = (lo_x + j) * kBN;
        // explicit key positions: the tile's 128 into this warp's copy in
        // shared memory (lane l loads columns l + 32 q) and their range, while
        // S is computed; keys past the end take a position after every query
        // (masked below)
        int* wpos = nullptr;
        int kmin = 0, kmax = 0;
        if constexpr (POS) {
          const int* kpos = p.key_pos + static_cast<size_t>(it.bh) * p.Lk;
          int kp[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int jj = j0 + 32 * q + lane;
            kp[q] = jj < p.Lk ? __ldg(kpos + jj) : 0x7fffffff;
          }
          wpos = reinterpret_cast<int*>(aux + fwd_aux_bytes(MODE, p) - 8u * 128u * 4u) + (warp - 4) * 128;
          __syncwarp();  // the previous tile's reads are done
#pragma unroll
          for (int q = 0; q < 4; ++q) wpos[32 * q + lane] = kp[q];
          kmin = __reduce_min_sync(0xffffffffu, min(min(kp[0], kp[1]), min(kp[2], kp[3])));
          kmax = __reduce_max_sync(0xffffffffu, max(max(kp[0], kp[1]), max(kp[2], kp[3])));
          __syncwarp();
        }
        bool ok = mbar_wait(bar(kBarSFull + x), cnt & 1);
        err = __any_sync(0xffffffffu, !ok);
        if (err) break;
        tc_fence_after();
        __syncwarp();

        uint32_t sr[4][32];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32(tS + q * 32, sr[q]);
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld_wait(sr[q]);
        tc_fence_before();
        mbar_arrive(bar(kBarSFree + x));  // the next S may overwrite this buffer
        float* xs = reinterpret_cast<float*>(&sr[0][0]);

        // ---- tile class, per warp (its 32 rows): far (one constant per row)
        // or near (per element). Deciding per warp rather than per tile lets
        // the warps of a tile next to the diagonal whose rows do not reach
        // the near band take the far path.
        const int p_lo_w = p_lo + 32 * (warp & 3);    // position of this warp's first row
        int rel_hi = j0 + kBN - 1 - p_lo_w;    // largest key - query offset in the warp's rows
        int rel_lo = j0 - (p_lo_w + 31);       // smallest
        if constexpr (POS) {
          rel_hi = kmax == 0x7fffffff ? 0x3fffffff : kmax - p_lo_w;
          rel_lo = kmin - (p_lo_w + 31);
        }
        bool far_l, far_r;
        if constexpr (MODE == 0) {
          far_l = rel_hi <= -p.t5_R;
          far_r = p.t5.bidir && rel_lo >= p.t5_R;
        } else if constexpr (MODE == 3 || MODE == 4) {
          far_l = far_r = false;  // ALiBi never saturates; Transformer-XL's term is in the scores
        } else {
          far_l = rel_hi <= -kc;
          far_r = rel_lo >= kc;
        }
        const bool need_mask = POS ? ((p.causal && rel_hi > 0) || (j0 + kBN > lk_eff))
                                   : ((p.causal && j0 + kBN - 1 > p_lo_w) || (j0 + kBN > lk_eff));
        int lim = 127;
        if (need_mask) {
          lim = lk_eff - 1 - j0;
          if (p.causal) lim = min(lim, prow - j0);
        }

        // Far tiles keep the raw scores s (logit = s * sl2 + addc, one constant
        // per row); near tiles get their per-element logits in place. Masking,
        // the maximum and the exponentials are then shared: the maximum is
        // taken on xs and mapped to logit units, and each probability is
        // 2^(xs * xscale + xoff - m).
        // DeBERTa tiles beyond the band still carry a per-key term, so every
        // DeBERTa tile takes the per-element path.
        // (explicit positions: a masked tile takes the per-element path,
        // unless every key is masked for every row of the warp: that tile
        // takes the far path with the constant -inf, all its probabilities 0)
        const bool dead = POS && ((p.causal && rel_lo > 0) || kmin == 0x7fffffff);
        const bool far =
            MODE == 3 || MODE == 4 || dead || (MODE != 2 && (far_l || far_r) && !(POS && need_mask));
        // a row constant added with the maximum: the far constant of a far
        // tile, for DeBERTa tiles beyond the band the saturated c2p term
        // (their per-key p2c term goes into the scaled scores), for ALiBi
        // tiles on one side of the diagonal the distance term of column 0
        // (a positions tile that takes the per-element path forms its whole
        // logit there)
        float addc = (far_l || far_r) && (far || !POS) ? (far_l ? add_l : add_r) : 0.f;
        if (dead) addc = kNegInf;
        if constexpr (MODE == 3) {
          // bias = -slope |r0 + c| with r0 = j0 - p the offset of column 0:
          // keys all ahead, -slope r0 - slope c; all behind, slope r0 + slope c;
          // a tile across the diagonal takes the whole term per column. The
          // column part goes into the raw scores in their own units (alibi_k
          // = slope / scale), which the exponent's FMA then scales.
          const float r0f = static_cast<float>(j0 - prow);
          if (rel_lo >= 0 || rel_hi <= 0) {
            const float sgn = rel_lo >= 0 ? -1.f : 1.f;
            addc = sgn * alibi_k * sl2 * r0f;
            const float2 cs2 = make_float2(sgn * alibi_k, sgn * alibi_k);
#pragma unroll
            for (int c = 0; c < 128; c += 2) {
              const float2 a = __ffma2_rn(make_float2(static_cast<float>(c), static_cast<float>(c + 1)), cs2,
                                          make_float2(xs[c], xs[c + 1]));
              xs[c] = a.x;
              xs[c + 1] = a.y;
            }
          } else {
            const float2 nk2 = make_float2(-alibi_k, -alibi_k);
#pragma unroll
            for (int c = 0; c < 128; c += 2) {
              const float2 dist = make_float2(fabsf(r0f + static_cast<float>(c)), fabsf(r0f + static_cast<float>(c + 1)));
              const float2 a = __ffma2_rn(dist, nk2, make_float2(xs[c], xs[c + 1]));
              xs[c] = a.x;
              xs[c + 1] = a.y;
            }
          }
        }
        if (!far) {
          if constexpr (POS) {
            // bias and mask per element from the keys' positions (offset key
            // position - query position; beyond the table's ends the buckets
            // are the saturated ones the ends hold)
            const float* tb = tab.copy(buf, 0);
            const int4* wp4 = reinterpret_cast<const int4*>(wpos);
#pragma unroll
            for (int q = 0; q < 32; ++q) {
              const int4 k4 = wp4[q];
              const int kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int c = 4 * q + e;
                const int rel = kk[e] == 0x7fffffff ? 0x3fffffff : kk[e] - prow;
                const float b = tb[min(max(rel + p.t5_tab_off, 0), p.t5_tab_len - 1)];
                const bool masked = (p.causal && rel > 0) || (j0 + c >= lk_eff);
                xs[c] = masked ? kNegInf : fmaf(xs[c], sl2, b);
              }
            }
          } else if (MODE == 0 && p.t5_compact) {
            const float* tb = tab.copy(buf, 0) + (j0 - prow + p.t5_tab_off);
#pragma unroll
            for (int c = 0; c < 128; ++c) xs[c] = fmaf(xs[c], sl2, tb[c]);
          } else if constexpr (MODE == 0) {
            const int s0 = j0 - prow + p.t5_tab_off;  // table index of column 0
            const int k = s0 & 3;
            const float4* tp = reinterpret_cast<const float4*>(tab.copy(buf, k) + (s0 - k));
            const float2 sc2 = make_float2(sl2, sl2);
#pragma unroll
            for (int q = 0; q < 32; ++q) {
              const float4 bq = tp[q];
              float2 a = make_float2(xs[4 * q], xs[4 * q + 1]);
              float2 b = make_float2(xs[4 * q + 2], xs[4 * q + 3]);
              a = __ffma2_rn(a, sc2, make_float2(bq.x, bq.y));
              b = __ffma2_rn(b, sc2, make_float2(bq.z, bq.w));
              xs[4 * q] = a.x;
              xs[4 * q + 1] = a.y;
              xs[4 * q + 2] = b.x;
              xs[4 * q + 3] = b.y;
            }
          } else if constexpr (MODE == 1) {
            const int r0 = j0 - prow;
#pragma unroll
            for (int c = 0; c < 128; ++c) {
              const int r = min(max(r0 + c, -kc), kc) + kc;
              xs[c] = fmaf(xs[c], sl2, qa[r]);
            }
          } else if constexpr (MODE == 2) {
            // the keys' saturated p2c values came with the tile's V stage
            // (ring position kv_it + its stream position; the stage is
            // released only after this tile's P.V, which waits for P)
            const uint32_t rpos = kv_it + static_cast<uint32_t>(it.split ? 2 * j + x : j);
            const uint32_t vst = rpos % kRing;
            const bool okv = mbar_wait(bar(kBarVFull + vst), (rpos / kRing) & 1);
            err = __any_sync(0xffffffffu, !okv);
            if (err) break;
            const float* ends_s = reinterpret_cast<const float*>(smem + kOffV + vst * L::kVBytes + kTileBytes);
            if (far_l || far_r) {
              // p2c: the saturated end column of every key; the c2p row
              // constant is addc
              const float4* ce = reinterpret_cast<const float4*>(ends_s + (far_l ? 0 : 128));
              const float2 sc2 = make_float2(sl2, sl2);
#pragma unroll
              for (int q = 0; q < 32; ++q) {
                const float4 e = ce[q];
                float2 a = __ffma2_rn(make_float2(xs[4 * q], xs[4 * q + 1]), sc2, make_float2(e.x, e.y));
                float2 b = __ffma2_rn(make_float2(xs[4 * q + 2], xs[4 * q + 3]), sc2, make_float2(e.z, e.w));
                xs[4 * q] = a.x;
                xs[4 * q + 1] = a.y;
                xs[4 * q + 2] = b.x;
                xs[4 * q + 3] = b.y;
              }
            } else {
              // band: column c is key j = j0 + c, at band offset m = j - i + k
              // = m0 + c. For 1 <= m <= 2k - 1 the row's band array holds
              // c2p + p2c; beyond, the far terms of its side apply. The window
              // starts 16-byte aligned (band_sh + m0 is a multiple of 8).
              const int m0 = j0 - prow + kc;
              const uint4* bw = reinterpret_cast<const uint4*>(band_row + (band_sh + m0));
              const float2 sc2 = make_float2(sl2, sl2);
              if (rel_lo > -kc && rel_hi < kc) {
                // the whole tile lies inside the band
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                  const uint4 u = __ldg(bw + q);
                  const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    const int c = 8 * q + 2 * e;
                    const float2 bv = make_float2(__uint_as_float(w4[e] << 16), __uint_as_float(w4[e] & 0xffff0000u));
                    const float2 a = __ffma2_rn(make_float2(xs[c], xs[c + 1]), sc2, bv);
                    xs[c] = a.x;
                    xs[c + 1] = a.y;
                  }
                }
              } else {
                const float4* e0 = reinterpret_cast<const float4*>(ends_s);
                const float4* e1 = e0 + 32;
                const int clo = 1 - m0, chi = 2 * kc - 1 - m0;  // in-band columns
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                  const uint4 u = __ldg(bw + q);
                  const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                  for (int g = 0; g < 2; ++g) {
                    const float4 f0 = e0[2 * q + g];
                    const float4 f1 = e1[2 * q + g];
                    const float l4[4] = {f0.x, f0.y, f0.z, f0.w};
                    const float r4[4] = {f1.x, f1.y, f1.z, f1.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                      const int c = 8 * q + 4 * g + e;
                      const uint32_t w = w4[2 * g + (e >> 1)];
                      const float bv = __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
                      const float far_v = c < clo ? add_l + l4[e] : add_r + r4[e];
                      xs[c] = fmaf(xs[c], sl2, (c >= clo && c <= chi) ? bv : far_v);
                    }
                  }
                }
              }
            }
          }
        }
        if (need_mask && !POS) {
#pragma unroll
          for (int c = 0; c < 128; ++c) xs[c] = (c > lim) ? kNegInf : xs[c];
        }
        float mx;
        {
          float m0 = kNegInf, m1 = kNegInf, m2 = kNegInf, m3 = kNegInf;
#pragma unroll
          for (int c = 0; c < 128; c += 8) {
            m0 = max3f(m0, xs[c], xs[c + 1]);
            m1 = max3f(m1, xs[c + 2], xs[c + 3]);
            m2 = max3f(m2, xs[c + 4], xs[c + 5]);
            m3 = max3f(m3, xs[c + 6], xs[c + 7]);
          }
          mx = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
          mx = far ? fmaf(mx, sl2, addc) : mx + addc;
        }
        if (STAG && x == 0 && j == 0) mbar_arrive(bar(kBarStag + (stag_it & 1)));

        // ---- running max with lazy rescale
        const float m_new = fmaxf(m_run, mx);
        const bool resc = m_new > m_run + kRescaleThreshold;
        float alpha = 1.f;
        if (resc) {
          alpha = ex2_approx(m_run - m_new);
          m_run = m_new;
        }
        const float m_use = (m_run == kNegInf) ? 0.f : m_run;

        // ---- probabilities, row sum, bf16 pack; x * 1 + c
        // is exact, so near tiles round exactly as a plain subtraction would
        uint32_t pk[64];
        float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
        {
          const float2 sc2 = far ? make_float2(sl2, sl2) : make_float2(1.f, 1.f);
          const float off = addc - m_use;
          const float2 off2 = make_float2(off, off);
#pragma unroll
          for (int c = 0; c < 128; c += 4) {
            float2 a = __ffma2_rn(make_float2(xs[c], xs[c + 1]), sc2, off2);
            float2 b = __ffma2_rn(make_float2(xs[c + 2], xs[c + 3]), sc2, off2);
            a.x = ex2_approx(a.x);
            a.y = ex2_approx(a.y);
            b.x = ex2_approx(b.x);
            b.y = ex2_approx(b.y);
            acc0 = __fadd2_rn(acc0, a);
            acc1 = __fadd2_rn(acc1, b);
            pk[c / 2] = pack_bf16x2(a.x, a.y);
            pk[c / 2 + 1] = pack_bf16x2(b.x, b.y);
          }
        }
        const float tile_sum = (acc0.x + acc0.y) + (acc1.x + acc1.y);
        l_run = l_run * alpha + tile_sum;

        // ---- the previous P.V of this tile must be done before P / O change
        if (cnt > 0) {
          ok = mbar_wait(bar(kBarODone + x), (cnt - 1) & 1);
          err = __any_sync(0xffffffffu, !ok);
          if (err) break;
          tc_fence_after();
        }
        __syncwarp();
        if (j > 0 && __any_sync(0xffffffffu, resc)) {
#pragma unroll
          for (int hc = 0; hc < DH / 64; ++hc) {
            uint32_t o[2][32];
            tmem_ld32(tO + 64 * hc, o[0]);
            tmem_ld32(tO + 64 * hc + 32, o[1]);
            tmem_ld_wait(o[0]);
            tmem_ld_wait(o[1]);
#pragma unroll
            for (int q = 0; q < 2; ++q)
#pragma unroll
              for (int c = 0; c < 32; ++c) o[q][c] = __float_as_uint(__uint_as_float(o[q][c]) * alpha);
            tmem_st32(tO + 64 * hc, o[0]);
            tmem_st32(tO + 64 * hc + 32, o[1]);
          }
        }
        tmem_st32(tP, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
        tmem_st32(tP + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(bar(kBarPFull + x));
        // Shaw: the value-side mass per clipped offset, after P is handed to
        // the tensor core (its P.V runs meanwhile)
        if constexpr (MODE == 1) {
          if (resc && j > 0) {
            for (int r = 0; r < nrel; ++r) wbin[r] *= alpha;
            mass_l *= alpha;
            mass_r *= alpha;
          }
          if (far_l) {
            mass_l += tile_sum;
          } else if (far_r) {
            mass_r += tile_sum;
          } else {
            // In-band offsets (-k < rel < k) into their bins, masses beyond
            // the clip in registers, from P as the P.V product takes it
            // (bf16, read back from TMEM). Each in-band (row, offset) pair
            // meets exactly one key of the item, so its bin is written once:
            // a plain (predicated) store, as the lanes (rows one offset
            // apart) disagree on which columns are in band. Only 16-column
            // chunks from one end of the tile through the warp's band are
            // read; the columns beyond lie on one side for every lane, and
            // their mass is the tile's sum less what was read. The rolled
            // chunk loop keeps this rarely taken path's code short.
            const int r0 = j0 - prow;
            const int rlo = 1 - kc - (j0 - p_lo_w);                  // lane 0's first in-band column
            const int chl = min(max(rlo, 0), 127) >> 4;                // chunks holding band columns
            const int chh = min(max(rlo + 29 + 2 * kc, 0), 127) >> 4;  // (lane 31's last: rlo + 31 + 2k - 2)
            const bool from_left = chh + 1 <= 8 - chl;                 // read [0, chh], else [chl, 7]
            const int ch0 = from_left ? 0 : chl, ch1 = from_left ? chh : 7;
            const uint32_t wb0 = smem_u32(wbin);
            float ml = 0.f, mr = 0.f, rd = 0.f;
#pragma unroll 1
            for (int ch = ch0; ch <= ch1; ++ch) {
              uint32_t w8[8];
              tmem_ld8_sync(tP + 8 * ch, w8);
#pragma unroll
              for (int e = 0; e < 16; ++e) {
                const int rel = r0 + 16 * ch + e;
                const float v = __uint_as_float((e & 1) ? (w8[e >> 1] & 0xffff0000u) : (w8[e >> 1] << 16));
                rd += v;
                ml += rel <= -kc ? v : 0.f;
                mr += rel >= kc ? v : 0.f;
                st_shared_f32_if(wb0 + 4u * static_cast<uint32_t>(min(max(rel + kc, 0), 2 * kc)), v,
                                 static_cast<unsigned>(rel + kc - 1) < static_cast<unsigned>(2 * kc - 1));
              }
            }
            const float rest = tile_sum - rd;  // the unread columns, all on the far side
            mass_l += from_left ? ml : ml + rest;
            mass_r += from_left ? mr + rest : mr;
          }
        }

      }
      if (err) break;
      if constexpr (MODE == 0) {
        // the next item's table, while the last P.V of this one runs
        if (next_h >= 0 && !t5_build((ocnt + 1) & 1)) {
          err = true;
          break;
        }
      }

      // ---- epilogue of this item
      {
        const bool ok = mbar_wait(bar(kBarODone + x), (cnt - 1) & 1);
        err = __any_sync(0xffffffffu, !ok);
        if (err) break;
      }
      tc_fence_after();
      __syncwarp();
      if constexpr (MODE == 1) {
        // the bins (with the masses beyond the clip) as the bf16 A operand of
        // O += bins . a_V, over this row's q . a_K values (no longer needed)
        wbin[0] += mass_l;
        wbin[2 * kc] += mass_r;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t w4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int r = 8 * c + 2 * e;
            w4[e] = pack_bf16x2(r < nrel ? wbin[r] : 0.f, r + 1 < nrel ? wbin[r + 1] : 0.f);
          }
          *reinterpret_cast<uint4*>(wb_tile + t * 128 + ((c ^ (t & 7)) << 4)) = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
        fence_async_smem();
        mbar_arrive(bar(kBarWb + x));
        const bool okv = mbar_wait(bar(kBarOv + x), ocnt & 1);
        err = __any_sync(0xffffffffu, !okv);
        if (err) break;
        tc_fence_after();
      }
      // A split item whose other half also has key tiles: merge the two
      // partial states. Each warpgroup publishes its rows' (m, l), then writes
      // 32 of the 64 output columns from both O accumulators, each scaled
      // from its own running maximum to the common one.
      const bool merge = it.split && sel(it.hi, x ^ 1) > sel(it.lo, x ^ 1);
      float sa = 1.f, sb = 0.f, l_row = l_run;
      if (merge) {
        // (one buffer suffices: the partner writes it again only after a P.V
        // that waits for this warpgroup's release of the accumulators below)
        float2* slot = ml;
        slot[x * 128 + t] = make_float2(m_run, l_run);
        mbar_arrive(bar(kBarComb));
        const bool ok = mbar_wait(bar(kBarComb), ccnt & 1);
        ++ccnt;
        err = __any_sync(0xffffffffu, !ok);
        if (err) break;
        tc_fence_after();
        const float2 other = slot[(x ^ 1) * 128 + t];
        const float m = fmaxf(m_run, other.x);
        sa = m_run == kNegInf ? 0.f : ex2_approx(m_run - m);
        sb = other.x == kNegInf ? 0.f : ex2_approx(other.x - m);
        l_row = l_run * sa + other.y * sb;
      }
      const int row = i0 + t;
      // rows past a padded element's length are zero rows
      const float inv_l = (l_row > 0.f && (!PAD || row < nlen)) ? 1.f / l_row : 0.f;
      // 64 columns at a time (32 of each accumulator when merging); the
      // accumulators are released after the last TMEM load
#pragma unroll
      for (int hc = 0; hc < DH / 64; ++hc) {
        const int c0 = merge ? x * (DH / 2) + 32 * hc : 64 * hc;
        uint32_t orr[2][32];
        if (merge) {
          tmem_ld32(tO + c0, orr[0]);
          tmem_ld32(tmem + lane_base + kTmemO + (x ^ 1) * DH + c0, orr[1]);
        } else {
          tmem_ld32(tO + c0, orr[0]);
          tmem_ld32(tO + c0 + 32, orr[1]);
        }
        tmem_ld_wait(orr[0]);
        tmem_ld_wait(orr[1]);
        if (hc == DH / 64 - 1) {
          tc_fence_before();
          // the next items' P.V may overwrite the accumulators read here
          mbar_arrive(bar(kBarOFree + x));
          mbar_arrive(bar(kBarOFree + (merge ? (x ^ 1) : x)));
          ++ocnt;
        }
        float* o = reinterpret_cast<float*>(&orr[0][0]);
        if (merge) {
#pragma unroll
          for (int c = 0; c < 32; ++c) o[c] = o[c] * sa + o[32 + c] * sb;
        }
        if (row < p.Lq) {
          const size_t base = (static_cast<size_t>(it.bh) * p.Lq + row) * DH + c0;
          const int ncol = merge ? 32 : 64;
          // each store instruction of a warp touches 32 rows, one line each:
          // 32-byte stores halve those line writes when the output allows them
          if constexpr (OUT_F32) {
            float* dst = static_cast<float*>(p.out) + base;
            auto w = [&](int c) { return __float_as_uint(o[c] * inv_l); };
            if (p.out_v8) {
#pragma unroll
              for (int c = 0; c < 64; c += 8)
                if (c < ncol)
                  st_global_v8(dst + c, w(c), w(c + 1), w(c + 2), w(c + 3), w(c + 4), w(c + 5), w(c + 6), w(c + 7));
            } else {
#pragma unroll
              for (int c = 0; c < 64; c += 4)
                if (c < ncol) st_global_v4(dst + c, w(c), w(c + 1), w(c + 2), w(c + 3));
            }
          } else {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.out) + base;
            auto w = [&](int c) { return pack_bf16x2(o[c] * inv_l, o[c + 1] * inv_l); };
            if (p.out_v8) {
#pragma unroll
              for (int c = 0; c < 64; c += 16)
                if (c < ncol)
                  st_global_v8(dst + c, w(c), w(c + 2), w(c + 4), w(c + 6), w(c + 8), w(c + 10), w(c + 12), w(c + 14));
            } else {
#pragma unroll
              for (int c = 0; c < 64; c += 8)
                if (c < ncol) st_global_v4(dst + c, w(c), w(c + 2), w(c + 4), w(c + 6));
            }
          }
        }
      }
    }
    if (err) {
      record_error(p.status);
      *abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

uint32_t fwd_smem_bytes(int mode, const FwdParams& p) {
  uint32_t aux0 = mode == 4   ? Smem<4>::kOffAux
                  : mode == 2 ? Smem<2>::kOffAux
                  : mode == 1 ? Smem<1>::kOffAux
                              : Smem<0>::kOffAux;
  static_assert(Smem<0>::kOffAux == Smem<3>::kOffAux, "T5 and ALiBi share the layout");
  if (p.dh == 128) aux0 = Smem<8>::kOffAux;  // T5 and ALiBi share the layout
  static_assert(Smem<8>::kOffAux == Smem<11>::kOffAux, "d = 128 layouts");
  return 1024u + aux0 + fwd_aux_bytes(mode, p) + (p.nsplit > 0 ? kCombBytes : 0u);
}

uint32_t fwd_max_smem_bytes() { return 232448u; }

int fwd_num_items(const FwdParams& p) { return p.B * p.H * p.npairs + p.nsplit; }

// The grid runs ceil(items / num_sms) passes. When the pair items left for the
// last pass fill at most half the grid, running each as two split items
// (half the key tiles per softmax warpgroup) halves that pass. This holds
// when every pair costs the same (no causal mask; causal items are ordered
// longest first, so the last pass's are the shortest and splitting them
// only unbalances the grid). A converted pair must hold two query tiles; the
// tail holds the lowest pair rows, and the highest converted row is checked.
int fwd_split_items(int npair_items, int BH, int Lq, int causal, int num_sms) {
  if (causal || num_sms <= 0 || npair_items <= 0) return 0;
  const int rem = npair_items % num_sms;
  if (rem == 0 || 2 * rem > num_sms) return 0;
  const int npairs = npair_items / BH;
  const int top_pair = npairs - 1 - (npair_items - rem) / BH;  // highest converted pair row
  if ((2 * top_pair + 1) * kBM >= Lq) return 0;
  return rem;
}

cudaError_t launch_fwd(int mode, bool out_f32, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                       const CUtensorMap& tmV, const CUtensorMap& tmS, const FwdParams& p, int num_sms,
                       cudaStream_t stream) {
  const uint32_t smem = fwd_smem_bytes(mode, p);
  const int nitems = fwd_num_items(p);
  dim3 grid(nitems < num_sms ? nitems : num_sms);
  dim3 block(kThreads);
  void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, const FwdParams) =
      nullptr;
  const int var = p.key_pos ? 4 : (p.lengths ? 3 : (p.nsplit > 0 ? 1 : (p.stagger ? 2 : 0)));
  // every mode has variants 0, 1 and 3; T5 and Transformer-XL also 2; d = 128
  // (T5 and ALiBi, bf16 output) has its own
#define RP_FWD_VARIANTS(M)                                                                         \
  if (var == 0) kern = out_f32 ? relpos_fwd_kernel<M, true, 0> : relpos_fwd_kernel<M, false, 0>;   \
  if (var == 1) kern = out_f32 ? relpos_fwd_kernel<M, true, 1> : relpos_fwd_kernel<M, false, 1>;   \
  if (var == 3) kern = out_f32 ? relpos_fwd_kernel<M, true, 3> : relpos_fwd_kernel<M, false, 3>;
  if (p.dh == 128) {
    if (out_f32 || (mode != 0 && mode != 3)) return cudaErrorNotSupported;
    if (mode == 0) {
      if (var == 0) kern = relpos_fwd_kernel<8, false, 0>;
      if (var == 1) kern = relpos_fwd_kernel<8, false, 1>;
      if (var == 2) kern = relpos_fwd_kernel<8, false, 2>;
      if (var == 3) kern = relpos_fwd_kernel<8, false, 3>;
    } else {
      if (var == 0) kern = relpos_fwd_kernel<11, false, 0>;
      if (var == 1) kern = relpos_fwd_kernel<11, false, 1>;
      if (var == 3) kern = relpos_fwd_kernel<11, false, 3>;
    }
  } else if (mode == 0) {
    RP_FWD_VARIANTS(0)
    if (var == 2) kern = out_f32 ? relpos_fwd_kernel<0, true, 2> : relpos_fwd_kernel<0, false, 2>;
    if (var == 4 && !out_f32) kern = relpos_fwd_kernel<0, false, 4>;
  } else if (mode == 1) {
    RP_FWD_VARIANTS(1)
  } else if (mode == 2) {
    RP_FWD_VARIANTS(2)
  } else if (mode == 3) {
    RP_FWD_VARIANTS(3)
  } else if (mode == 4) {
    RP_FWD_VARIANTS(4)
    if (var == 2) kern = out_f32 ? relpos_fwd_kernel<4, true, 2> : relpos_fwd_kernel<4, false, 2>;
  }
#undef RP_FWD_VARIANTS
  if (!kern) return cudaErrorNotSupported;
  // raise the kernel's shared-memory limit once per device (the maximum, so
  // that every later launch fits)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  const int slot = (p.dh == 128 ? 5 + (mode == 3 ? 1 : 0) : mode) * 16 + (out_f32 ? 8 : 0) + var;
  static std::atomic<uint64_t> attr_set[7 * 16];
  const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
  if (!bit || !(attr_set[slot].load() & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(fwd_max_smem_bytes()));
    if (e != cudaSuccess) return e;
    attr_set[slot].fetch_or(bit);
  }
  // programmatic dependent launch: the setup of this launch may overlap the
  // end of the previous kernel in the stream (the kernel waits for it before
  // its first global-memory access)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tmQ, tmK, tmV, tmS, p);
}

}  // namespace relpos
