// sgemv_m1.cu -- SparseGemv for one activation row (m = 1, decode).
//
// Product (Dong et al., arXiv 2605.11582, section 1 contribution 2 and
// section 3.3): y[r] = sum over kept j of (q_j - z) * s * x[4 quad(j) + pos_j],
// fp32 accumulation, one rounding to binary16 per output.
//
// The work is bound by HBM bandwidth on the packed weight (0.81 bytes per
// kept weight), so the kernel keeps many bytes in flight and issues few
// instructions per weight:
//
//  * Weights stream through a per-warp ring of two shared-memory stages
//    filled by asynchronous copies (cp.async): each lane copies its 16 bytes
//    of nibbles, 8 bytes of codes and its scale/zero word for the item two
//    ahead into a region only it reads, so no registers hold data in flight
//    and no cross-lane synchronisation is needed.  A row of a K slice is a
//    fixed number of items (1 to 4, a template parameter), so copy offsets
//    and table offsets are constants of the unrolled row, and so are the
//    ring stages when the row is a whole number of rings.  The first stages
//    are issued before the programmatic-dependent-launch wait, overlapping
//    the previous kernel.  (Per-warp bulk TMA copies of the same stages were
//    measured slower: the items are 128-512 B, too small for the TMA unit.)
//  * Pair tables of x in shared memory.  A "pair unit" is two kept weights
//    whose columns are fixed by one stored 4-bit position field (2:4: the
//    quad's two positions, 6 values; 1:4: two adjacent quads' positions, 16
//    values).  For
//    every unit the table holds all candidate (x_first, x_second) pairs as
//    fp32, so one 8-byte shared load fetches both activations already
//    widened.  Each lane owns a private bank column (8 bytes of every
//    128-byte line), so the data-dependent lookups never conflict.
//  * INT4 decode by the exponent trick: OR-ing a nibble shifted by p into
//    the mantissa of 2^23 gives the float 2^23 + q 2^p; subtracting
//    2^23 + z 2^p is exact and leaves (q - z) 2^p.  Each byte of a word is a
//    pair unit; bytes 0, 1 decode in place, bytes 2, 3 after one shift; the
//    2^p factors are removed once per chunk.
//  * Packed f32x2 arithmetic (sm_100+) for the subtract and the FMA.
//  * Large K is cut into slices that fit the table; row partial sums carry
//    over slices in shared memory.
#include <string.h>

#include "sgemv_internal.cuh"

namespace sgemv {
namespace {

#ifndef SGEMV_M1_NT
#define SGEMV_M1_NT 512
#endif
#ifndef SGEMV_M1_NT_MANY
#define SGEMV_M1_NT_MANY 640
#endif
#ifndef SGEMV_M1_D
#define SGEMV_M1_D 2
#endif
#ifndef SGEMV_M1_STATIC
#define SGEMV_M1_STATIC 2
#endif
// Ring stages as constants: 2 = where a row is a whole number of rings
// (measured best: the smaller loop body of the grouped launches wins); 1 =
// also by unrolling rows; 0 = never.
constexpr int kStaticStages = SGEMV_M1_STATIC;
// Items in flight per warp: item t of a warp's stream sits in ring stage
// t % kS, and consuming it issues item t + kS.
constexpr int kS = SGEMV_M1_D;
static_assert(kS == 2 || kS == 4 || kS == 8, "ring stages: a power of two");
constexpr int kStage = 1024;        // bytes per stage
constexpr int kIdxOff = 512;        // codes after the 512 B of nibbles
constexpr int kSzOff = 768;         // scale/zero words after the codes
constexpr int kSmemLimit = 227 * 1024;
#ifndef SGEMV_M1_PREFETCH_X
#define SGEMV_M1_PREFETCH_X 1
#endif
constexpr bool kPrefetchX = SGEMV_M1_PREFETCH_X != 0;   // L2 prefetch of x before the wait
constexpr uint32_t kTabAlign = 2048;

// Pair-table geometry.  A unit's code indexes its entries at a 128-byte
// stride (one 8-byte pair per lane of a half-warp).  1:4: 16 codes, 16
// entries per unit.  2:4: the code is the stored position nibble a | b << 2,
// one of {4, 8, 9, 12, 13, 14}; entries sit at (code - 4) from the unit's
// base with units 7 entries apart -- the six codes are distinct mod 7, so
// units interleave without overlap (112 slots per chunk, padded to 128).
template <int N>
struct M1Cfg {
  static constexpr int E = N == 2 ? 7 : 16;          // unit stride in entries
  static constexpr int OFF0 = N == 2 ? -4 * 128 : 0; // entry of code 0 from the unit base
  static constexpr int SLOTS = N == 2 ? 128 : 256;   // entries per chunk (a multiple of 16)
  static constexpr int CPC = N == 2 ? 64 : 128;      // dense columns per chunk
  static constexpr int UC = N == 2 ? 4 : 8;          // dense columns per unit
  static constexpr int XPAD = CPC + 2;               // staged x per chunk (halves)
  // shared bytes per chunk-per-lane of a K slice
  static constexpr int TAB_PER_CPL = 32 * SLOTS * 8;
  static constexpr int X_PER_CPL = 32 * XPAD * 2;
};

// The six position nibbles a | b << 2 (a < b) of a 2:4 quad.
__device__ __forceinline__ constexpr int quad24_nibble(int e) {
  return e == 0 ? 0x4 : e == 1 ? 0x8 : e == 2 ? 0xC : e == 3 ? 0x9 : e == 4 ? 0xD : 0xE;
}

// One packed matrix of a launch.  A launch covers up to kMaxSeg matrices
// that share x (and N): their rows are concatenated into one row space.
constexpr int kMaxSeg = 8;
struct M1Seg {
  const uint4* vals;
  const uint2* idx;
  const uint32_t* sz;
  __half* y;
  int row_begin;     // first row of this matrix in the launch's row space
  int gstride;       // scale/zero words per row in memory
  int gshift;        // log2(group)
  int g64;           // 1:4 with 64-column groups: two groups per chunk
};

struct M1Params {
  M1Seg seg[kMaxSeg];
  int nseg;
  const __half* x;
  int* err;
  int rows, cols;    // rows of all matrices together
  int chunks;        // chunks holding a row's kept weights
  int cstride;       // chunks per row in memory
  int rows_per_cta;
  int slice_chunks;  // 32 * cpl
  int nslices;
  int cpl;
};

__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;");
}

// dst + DOFF <- src + SOFF (bytes), issued only where `on` is set when PRED
// (a predicated instruction, so lanes without a chunk need no branch).
template <int BYTES, int DOFF, int SOFF, bool PRED>
__device__ __forceinline__ void cp_async_at(bool on, uint32_t dst, const void* src) {
  if constexpr (PRED) {
    if constexpr (BYTES == 16)
      asm volatile(
          "{ .reg .pred p; setp.ne.b32 p, %2, 0; @p cp.async.cg.shared.global [%0+%3], [%1+%4], 16; }" ::"r"(dst),
          "l"(src), "r"((int)on), "n"(DOFF), "n"(SOFF)
          : "memory");
    else
      asm volatile(
          "{ .reg .pred p; setp.ne.b32 p, %2, 0; @p cp.async.ca.shared.global [%0+%3], [%1+%4], %5; }" ::"r"(dst),
          "l"(src), "r"((int)on), "n"(DOFF), "n"(SOFF), "n"(BYTES)
          : "memory");
  } else {
    if constexpr (BYTES == 16)
      asm volatile("cp.async.cg.shared.global [%0+%2], [%1+%3], 16;" ::"r"(dst), "l"(src), "n"(DOFF),
                   "n"(SOFF)
                   : "memory");
    else
      asm volatile("cp.async.ca.shared.global [%0+%2], [%1+%3], %4;" ::"r"(dst), "l"(src), "n"(DOFF),
                   "n"(SOFF), "n"(BYTES)
                   : "memory");
  }
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int OFF>
__device__ __forceinline__ uint4 lds128_at(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4+%5];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a), "n"(OFF));
  return v;
}
template <int OFF>
__device__ __forceinline__ uint2 lds64_at(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2+%3];" : "=r"(v.x), "=r"(v.y) : "r"(a), "n"(OFF));
  return v;
}

template <int OFF>
__device__ __forceinline__ float2 lds_pair(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0,%1}, [%2+%3];"
               : "=f"(v.x), "=f"(v.y)
               : "r"(addr), "n"(OFF));
  return v;
}

__device__ __forceinline__ void sts_pair(uint32_t addr, float a, float b) {
  asm volatile("st.shared.v2.f32 [%0], {%1,%2};" ::"r"(addr), "f"(a), "f"(b));
}


// Subtract constants for one (scale, zero) group: -(2^23 + z 2^p) for the
// nibble classes p = (0, 4) and (8, 12).
struct ZConst {
  float2 ca, cb;
};

__device__ __forceinline__ ZConst zconst(float z) {
  const float2 zz = make_float2(z, z);
  const float2 mm = make_float2(-8388608.0f, -8388608.0f);
  ZConst k;
  k.ca = __ffma2_rn(zz, make_float2(-1.0f, -16.0f), mm);
  k.cb = __ffma2_rn(zz, make_float2(-256.0f, -4096.0f), mm);
  return k;
}

// 2^23 + q 2^p as a float, from the nibble at bits p..p+3 of v: one LOP3
// ((v & MASK) | magic) with the exponent pattern held in a register.
template <uint32_t MASK>
__device__ __forceinline__ float mag(uint32_t v, uint32_t magic) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(v), "n"(MASK), "r"(magic));
  return __uint_as_float(r);
}

// One 32-bit word of nibbles (pair units U0..U0+3, one per byte) times its
// x pairs.  Bytes 0 and 1 decode in place (classes 2^0,2^4 and 2^8,2^12);
// bytes 2 and 3 after a 16-bit shift, into the same classes.
template <int E, int OFF0, int U0, bool FIRST>
__device__ __forceinline__ void word_fma(uint32_t v, uint32_t codes, uint32_t base,
                                         uint32_t magic, const ZConst& k, float2& a0,
                                         float2& a1, float2& a2, float2& a3) {
  const uint32_t vs = v >> 16;
  float2 d0 = make_float2(mag<0xFu>(v, magic), mag<0xF0u>(v, magic));
  float2 d1 = make_float2(mag<0xF00u>(v, magic), mag<0xF000u>(v, magic));
  float2 d2 = make_float2(mag<0xFu>(vs, magic), mag<0xF0u>(vs, magic));
  float2 d3 = make_float2(mag<0xF00u>(vs, magic), mag<0xF000u>(vs, magic));
  d0 = __fadd2_rn(d0, k.ca);
  d1 = __fadd2_rn(d1, k.cb);
  d2 = __fadd2_rn(d2, k.ca);
  d3 = __fadd2_rn(d3, k.cb);
  // code of unit U0+s sits at bits 4s of `codes`; table stride 128 B/entry
  const float2 x0 = lds_pair<OFF0 + (U0 + 0) * E * 128>(((codes << 7) & 0x780u) | base);
  const float2 x1 = lds_pair<OFF0 + (U0 + 1) * E * 128>(((codes << 3) & 0x780u) | base);
  const float2 x2 = lds_pair<OFF0 + (U0 + 2) * E * 128>(((codes >> 1) & 0x780u) | base);
  const float2 x3 = lds_pair<OFF0 + (U0 + 3) * E * 128>(((codes >> 5) & 0x780u) | base);
  if (FIRST) {
    a0 = __fmul2_rn(d0, x0);
    a1 = __fmul2_rn(d1, x1);
    a2 = __fmul2_rn(d2, x2);
    a3 = __fmul2_rn(d3, x3);
  } else {
    a0 = __ffma2_rn(d0, x0, a0);
    a1 = __ffma2_rn(d1, x1, a1);
    a2 = __ffma2_rn(d2, x2, a2);
    a3 = __ffma2_rn(d3, x3, a3);
  }
}

// Removes the 2^p class factors and folds the accumulators into one float:
// a0, a2 hold classes (2^0, 2^4), a1, a3 hold (2^8, 2^12).
__device__ __forceinline__ float fold(float2 a0, float2 a1, float2 a2, float2 a3) {
  const float2 lo = __fadd2_rn(a0, a2);
  const float2 hi = __fadd2_rn(a1, a3);
  float2 t = __fmul2_rn(lo, make_float2(1.0f, 0.0625f));
  t = __ffma2_rn(hi, make_float2(0x1p-8f, 0x1p-12f), t);
  return t.x + t.y;
}

__device__ __forceinline__ float sz_scale(uint32_t w) {
  return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu)));
}
__device__ __forceinline__ float sz_zero(uint32_t w) {
  return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
}

// acc plus the contribution of one chunk (32 kept weights) of one row, the
// group scale applied by explicit FMAs so that a row rounds the same way in
// every launch mode.  G2: the chunk spans two (scale, zero) groups (1:4 with
// 64-column groups), units 0..7 in the first and 8..15 in the second.
// TOFF: byte offset of the chunk's table slot from `base`.
template <int N, bool G2, int TOFF>
__device__ __forceinline__ float chunk_dot(const uint4& v, const uint2& ix,
                                           uint32_t sa, uint32_t sb, uint32_t base,
                                           uint32_t magic, float acc) {
  constexpr int E = M1Cfg<N>::E, O = M1Cfg<N>::OFF0 + TOFF;
  float2 a0, a1, a2, a3;
  if (!G2) {
    const ZConst k = zconst(sz_zero(sa));
    word_fma<E, O, 0, true>(v.x, ix.x, base, magic, k, a0, a1, a2, a3);
    word_fma<E, O, 4, false>(v.y, ix.x >> 16, base, magic, k, a0, a1, a2, a3);
    word_fma<E, O, 8, false>(v.z, ix.y, base, magic, k, a0, a1, a2, a3);
    word_fma<E, O, 12, false>(v.w, ix.y >> 16, base, magic, k, a0, a1, a2, a3);
    return fmaf(sz_scale(sa), fold(a0, a1, a2, a3), acc);
  } else {
    const ZConst ka = zconst(sz_zero(sa));
    word_fma<E, O, 0, true>(v.x, ix.x, base, magic, ka, a0, a1, a2, a3);
    word_fma<E, O, 4, false>(v.y, ix.x >> 16, base, magic, ka, a0, a1, a2, a3);
    const float ya = fmaf(sz_scale(sa), fold(a0, a1, a2, a3), acc);
    const ZConst kb = zconst(sz_zero(sb));
    word_fma<E, O, 8, true>(v.z, ix.y, base, magic, kb, a0, a1, a2, a3);
    word_fma<E, O, 12, false>(v.w, ix.y >> 16, base, magic, kb, a0, a1, a2, a3);
    return fmaf(sz_scale(sb), fold(a0, a1, a2, a3), ya);
  }
}

// MODE of a launch: kOne = one matrix, groups of 64 columns not split
// across chunks; kOneG64 = one 1:4 matrix with 64-column groups (two groups
// per chunk); kMany = several matrices, the split decided per row.
constexpr int kOne = 0, kOneG64 = 1, kMany = 2;

// Threads per CTA (one CTA per SM) of a launch mode: 20 warps for the
// grouped launches, 16 for one matrix (each measured the faster there; at
// 640 threads the kernel fits in under 100 registers without spilling).
template <int MODE>
constexpr int kNTm = MODE == kMany ? SGEMV_M1_NT_MANY : SGEMV_M1_NT;
template <int MODE>
constexpr int kNWm = kNTm<MODE> / 32;

// Rows of a CTA interleave over its warps: the warp's j-th row is local row
// warp + kNW j.
template <int MODE>
__device__ __forceinline__ int warp_nrows(int warp, int nr) {
  constexpr int kNW = kNWm<MODE>;
  return warp < nr ? (nr - warp + kNW - 1) / kNW : 0;
}

// Matrix of launch row `row`, searched forward from `seg` (a warp visits its
// rows in increasing order within a K slice).
template <int MODE>
__device__ __forceinline__ int seg_from(const M1Params& p, int seg, int row) {
  if (MODE == kMany)
    while (seg + 1 < p.nseg && row >= p.seg[seg + 1].row_begin) ++seg;
  return MODE == kMany ? seg : 0;
}

// The copy side of a warp's weight stream over one K slice.  It stands at
// row P of the warp (ordinal `pr`, launch row `row`) with per-lane pointers
// to the lane's chunk c0 + lane of each stream; item k of the row holds the
// chunks 32 k further on.
template <int N, int MODE>
struct RowProducer {
  const uint4* vp;     // nibbles, codes and scale/zero of item 0 of row P
  const uint2* ip;
  const uint32_t* sp;
  int sstep;           // scale/zero words between a lane's chunks in consecutive items
  int sstep_row;       // scale/zero words from row P to row P + kNW (same matrix)
  int vstep;           // chunks from row P to row P + kNW
  int next_begin;      // first launch row of the next matrix (kMany)
  int seg, pr, row;
  bool g64;            // two scale/zero words per chunk
  const M1Params* p_;  // (checked build)

  __device__ __forceinline__ void set_row(const M1Params& p, int c0, int lane) {
    using C = M1Cfg<N>;
    p_ = &p;
    seg = seg_from<MODE>(p, seg, row);
    const M1Seg& sg = p.seg[seg];
    const int lr = row - sg.row_begin;
    const int ch = c0 + lane;
    vp = sg.vals + (size_t)lr * p.cstride + ch;
    ip = sg.idx + (size_t)lr * p.cstride + ch;
    sp = sg.sz + (size_t)lr * sg.gstride + ((ch * C::CPC) >> sg.gshift);
    sstep = (32 * C::CPC) >> sg.gshift;
    g64 = N == 1 && (MODE == kMany ? sg.g64 != 0 : MODE == kOneG64);
    vstep = kNWm<MODE> * p.cstride;
    sstep_row = kNWm<MODE> * sg.gstride;
    next_begin = MODE == kMany && seg + 1 < p.nseg ? p.seg[seg + 1].row_begin : 0x7fffffff;
  }
  __device__ __forceinline__ void start(const M1Params& p, int r0, int warp, int c0, int lane) {
    pr = 0;
    row = r0 + warp;
    seg = 0;
    set_row(p, c0, lane);
  }
  // to the warp's next row (pointers only while it has one)
  __device__ __forceinline__ void advance(const M1Params& p, int c0, int lane, int nrw) {
    ++pr;
    row += kNWm<MODE>;
    if (pr >= nrw) return;
    if (row < next_begin) {
      vp += vstep;
      ip += vstep;
      sp += sstep_row;
    } else {
      set_row(p, c0, lane);
    }
  }
  // Copies this lane's part of item K of row P into the ring stage at
  // s16 + SO (nibbles) and s8 + SO (codes, scale/zero): 16 bytes of nibbles,
  // 8 bytes of codes and the scale/zero word(s), each into a region only
  // this lane reads.  PRED: only where `on` (the last item of a ragged
  // slice).
  template <int K, bool PRED, int SO>
  __device__ __forceinline__ void issue(uint32_t s16, uint32_t s8, bool on) const {
    const uint32_t* s = sp + K * sstep;
    if (!check(vp + 32 * K, s, !PRED || on)) return;
    cp_async_at<16, SO, K * 512, PRED>(on, s16, vp);
    cp_async_at<8, SO + kIdxOff, K * 256, PRED>(on, s8, ip);
    if (g64)
      cp_async_at<8, SO + kSzOff, 0, PRED>(on, s8, s);
    else
      cp_async_at<4, SO + kSzOff, 0, PRED>(on, s8, s);
  }
  // The same with K and the stage at run time (the prologue).
  __device__ __forceinline__ void issue_rt(int k, uint32_t s16, uint32_t s8, bool on) const {
    const uint32_t* s = sp + k * sstep;
    if (!check(vp + 32 * k, s, on)) return;
    cp_async_at<16, 0, 0, true>(on, s16, vp + 32 * k);
    cp_async_at<8, kIdxOff, 0, true>(on, s8, ip + 32 * k);
    if (g64)
      cp_async_at<8, kSzOff, 0, true>(on, s8, s);
    else
      cp_async_at<4, kSzOff, 0, true>(on, s8, s);
  }
  // (checked build) the chunk at v and its scale/zero word(s) at s lie
  // inside row P; false after recording an error
  __device__ __forceinline__ bool check(const uint4* v, const uint32_t* s, bool on) const {
    if constexpr (kChecked) {
      const M1Seg& sg = p_->seg[seg];
      const int64_t ch = v - (sg.vals + (size_t)(row - sg.row_begin) * p_->cstride);
      const int64_t gw = s - (sg.sz + (size_t)(row - sg.row_begin) * sg.gstride);
      if (on && (ch < 0 || ch >= p_->cstride || gw < 0 || gw + (g64 ? 1 : 0) >= sg.gstride)) {
        report_checked(p_->err);
        return false;
      }
    }
    return true;
  }
};

// What one warp's item loop over a K slice needs.
template <int N, int MODE>
struct SliceCtx {
  RowProducer<N, MODE>* prod;
  const M1Params* p;
  uint32_t ring16, ring8;   // this lane's regions of ring stage 0
  uint32_t lane_base;       // this lane's table column, chunk slot 0
  uint32_t magic;
  uint32_t par;             // (stages at run time) ring offset of the row's first item
  int c0, nrw, lane;
  bool last_on;             // this lane holds a chunk in the row's last item
};

// Item I of the current row (IPR items per row): waits for its copies,
// reads its ring stage, refills that stage with the item kS ahead in the
// warp's stream and adds the chunk's contribution to acc.  SO0: the stage
// of the row's item 0 when it is known at compile time, else -1 (c.par).
template <int N, int MODE, int IPR, int SO0, int I>
__device__ __forceinline__ void row_items(SliceCtx<N, MODE>& c, bool g64, float& acc) {
  if constexpr (I < IPR) {
    using C = M1Cfg<N>;
    constexpr bool kRt = SO0 < 0;
    constexpr int SO = kRt ? 0 : ((SO0 + I) % kS) * kStage;
    uint32_t r16 = c.ring16, r8 = c.ring8;
    if constexpr (kRt) {
      const uint32_t so = (c.par + I * kStage) & (kS * kStage - 1);
      r16 += so;
      r8 += so;
    }
    constexpr bool kLast = I == IPR - 1;
    const bool valid = !kLast || c.last_on;
    cp_wait<kS - 1>();   // this lane's copies of this item landed
    const uint4 v = lds128_at<SO>(r16);
    uint2 ix = lds64_at<SO + kIdxOff>(r8);
    if constexpr (kChecked && N == 2) {
      if (valid && (bad_codes24(ix.x) | bad_codes24(ix.y))) {
        report_checked(c.p->err);
        ix = make_uint2(0x44444444u, 0x44444444u);
      }
    }
    const uint2 s2 = lds64_at<SO + kSzOff>(r8);
    const uint32_t sa = valid ? s2.x : 0u;   // ragged slice: zero contribution
    const uint32_t sb = valid ? s2.y : 0u;
    // refill this stage with the item kS ahead: item K of a later row
    RowProducer<N, MODE>& q = *c.prod;
    constexpr int K = (I + kS) % IPR;
    if constexpr (K == 0) q.advance(*c.p, c.c0, c.lane, c.nrw);
    if (q.pr < c.nrw) q.template issue<K, K == IPR - 1, SO>(r16, r8, c.last_on);
    cp_commit();
    constexpr int TOFF = I * C::SLOTS * 128;
    if constexpr (N == 1 && MODE == kMany) {
      if (g64)
        acc = chunk_dot<N, true, TOFF>(v, ix, sa, sb, c.lane_base, c.magic, acc);
      else
        acc = chunk_dot<N, false, TOFF>(v, ix, sa, sb, c.lane_base, c.magic, acc);
    } else {
      acc = chunk_dot<N, N == 1 && MODE == kOneG64, TOFF>(v, ix, sa, sb, c.lane_base, c.magic,
                                                          acc);
    }
    row_items<N, MODE, IPR, SO0, I + 1>(c, g64, acc);
  }
}

// The first kS items of a slice's stream into the ring, one commit group
// each (empty past the warp's rows).  The producer is left on the row of
// the last item issued.
template <int N, int MODE>
__device__ __forceinline__ void stream_prologue(RowProducer<N, MODE>& prod, const M1Params& p,
                                                int r0, int warp, int lane, int c0, int ipr,
                                                int nrw, bool last_on, uint32_t ring16,
                                                uint32_t ring8) {
  if (nrw > 0) prod.start(p, r0, warp, c0, lane);
  int k = 0;
#pragma unroll
  for (int t = 0; t < kS; ++t) {
    if (nrw > 0) {   // (a warp without rows never starts its producer)
      if (t > 0 && k == 0) prod.advance(p, c0, lane, nrw);
      if (prod.pr < nrw)
        prod.issue_rt(k, ring16 + t * kStage, ring8 + t * kStage, k < ipr - 1 || last_on);
    }
    cp_commit();
    k = k + 1 == ipr ? 0 : k + 1;
  }
}

// One row of the warp (ordinal j): its IPR items, the warp reduction and
// the store.
template <int N, int MODE, int IPR, int SO0>
__device__ __forceinline__ void one_row(SliceCtx<N, MODE>& c, int r0, int warp, int j, int sl,
                                        float* part, int& seg) {
  const M1Params& p = *c.p;
  const int lr = warp + kNWm<MODE> * j;
  const int row = r0 + lr;
  seg = seg_from<MODE>(p, seg, row);
  const M1Seg& sg = p.seg[seg];
  const bool g64 = N == 1 && (MODE == kMany ? sg.g64 != 0 : MODE == kOneG64);
  float acc = 0.0f;
  row_items<N, MODE, IPR, SO0, 0>(c, g64, acc);
  if constexpr (SO0 < 0) c.par = (c.par + IPR * kStage) & (kS * kStage - 1);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (c.lane == 0) {
    __half* yrow = sg.y + (row - sg.row_begin);
    if (p.nslices == 1) {
      *yrow = __float2half_rn(acc);
    } else {
      const float t = (sl ? part[lr] : 0.0f) + acc;
      if (sl == p.nslices - 1)
        *yrow = __float2half_rn(t);
      else
        part[lr] = t;
    }
  }
}

// Rows j .. j + RU - 1 of the warp (those it has), unrolled so that the
// ring stage of every item is a constant.
template <int N, int MODE, int IPR, int RU, int JJ>
__device__ __forceinline__ void row_group(SliceCtx<N, MODE>& c, int r0, int warp, int j, int sl,
                                          float* part, int& seg) {
  if constexpr (JJ < RU) {
    if (JJ == 0 || j + JJ < c.nrw) {
      constexpr bool kStatic = kStaticStages == 1 ? (IPR % kS == 0 || kS % IPR == 0)
                                               : kStaticStages == 2 && IPR % kS == 0;
      one_row<N, MODE, IPR, kStatic ? (JJ * IPR) % kS : -1>(c, r0, warp, j + JJ, sl, part, seg);
      row_group<N, MODE, IPR, RU, JJ + 1>(c, r0, warp, j, sl, part, seg);
    }
  }
}

// A row's total (CTA row lr of matrix seg) into y, or into the partial
// carried over K slices.
__device__ __forceinline__ void store_row(const M1Params& p, int seg, int r0, int lr, int sl,
                                          float* part, float v) {
  const M1Seg& sg = p.seg[seg];
  __half* yrow = sg.y + (r0 + lr - sg.row_begin);
  if (p.nslices == 1) {
    *yrow = __float2half_rn(v);
  } else {
    const float t = (sl ? part[lr] : 0.0f) + v;
    if (sl == p.nslices - 1)
      *yrow = __float2half_rn(t);
    else
      part[lr] = t;
  }
}

// Rows of one item (IPR = 1), two at a time: one exchange across the
// half-warps leaves row j's partials in lanes 0..15 and row j + 1's in lanes
// 16..31, and four more butterfly steps finish both (the same additions,
// pair for pair, as a butterfly over each row alone).
template <int N, int MODE>
__device__ __forceinline__ void stream_rows_paired(SliceCtx<N, MODE>& c, int r0, int warp,
                                                   int sl, float* part) {
  const M1Params& p = *c.p;
  const bool hi = (c.lane & 16) != 0;
  int seg = 0;
  auto row_acc = [&](int j) -> float {
    const int row = r0 + warp + kNWm<MODE> * j;
    seg = seg_from<MODE>(p, seg, row);
    const M1Seg& sg = p.seg[seg];
    const bool g64 = N == 1 && (MODE == kMany ? sg.g64 != 0 : MODE == kOneG64);
    float acc = 0.0f;
    row_items<N, MODE, 1, -1, 0>(c, g64, acc);
    c.par ^= kStage;
    return acc;
  };
  for (int j = 0; j < c.nrw; j += 2) {
    const float a0 = row_acc(j);
    const int seg0 = seg;
    if (j + 1 < c.nrw) {
      const float a1 = row_acc(j + 1);
      float v = (hi ? a1 : a0) + __shfl_xor_sync(0xffffffffu, hi ? a0 : a1, 16);
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if ((c.lane & 15) == 0)
        store_row(p, hi ? seg : seg0, r0, warp + kNWm<MODE> * (j + (hi ? 1 : 0)), sl, part, v);
    } else {
      float v = a0;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (c.lane == 0) store_row(p, seg0, r0, warp + kNWm<MODE> * j, sl, part, v);
    }
  }
}

#ifndef SGEMV_M1_PAIR1
#define SGEMV_M1_PAIR1 1
#endif

// The warp's rows of one K slice, IPR items each.
template <int N, int MODE, int IPR>
__device__ __forceinline__ void stream_slice(SliceCtx<N, MODE>& c, int r0, int warp, int sl,
                                             float* part) {
  constexpr bool kStatic = kStaticStages == 1 ? (IPR % kS == 0 || kS % IPR == 0)
                                               : kStaticStages == 2 && IPR % kS == 0;
  if constexpr (IPR == 1 && !kStatic && SGEMV_M1_PAIR1 && MODE != kMany) {
    // a one-item row is short: reducing two rows together saves a fifth of
    // the reduction per row (single-matrix launches only: in the grouped
    // kernels the larger body cost more than it saved)
    stream_rows_paired<N, MODE>(c, r0, warp, sl, part);
  } else {
    constexpr int RU = kStatic && IPR < kS ? kS / IPR : 1;
    int seg = 0;
    for (int j = 0; j < c.nrw; j += RU) row_group<N, MODE, IPR, RU, 0>(c, r0, warp, j, sl, part, seg);
  }
}

// Items per row the kernel is compiled for: 2:4 slices of up to 128
// chunks, 1:4 of up to 64 (the pair tables of larger slices do not fit).
template <int N>
constexpr int max_ipr() { return N == 2 ? 4 : 2; }

// The body of one CTA; `cta` is its index within the launch part that
// covers these matrices (a launch may hold two parts, one per N).
template <int N, int MODE>
__device__ __forceinline__ void m1_body(const M1Params& p, int cta) {
  using C = M1Cfg<N>;
  extern __shared__ __align__(128) unsigned char smem[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int S = p.cpl * C::SLOTS;                  // table slots per half-warp
  const int tab_bytes = 2 * S * 128;
  // The table starts on a 2 KB boundary so that bits 7..10 of every slot
  // address come from the code alone (the lookups OR the code in).
  const uint32_t raw_s = (uint32_t)__cvta_generic_to_shared(smem);
  const uint32_t pad = (kTabAlign - (raw_s & (kTabAlign - 1))) & (kTabAlign - 1);
  unsigned char* tab = smem + pad;
  const uint32_t smem_s = raw_s + pad;
  const int xs_bytes = p.slice_chunks * C::XPAD * 2;
  __half* xs = reinterpret_cast<__half*>(tab + tab_bytes);
  float* part = reinterpret_cast<float*>(tab + tab_bytes + xs_bytes);
  const int part_bytes = (p.nslices > 1 ? (p.rows_per_cta * 4 + 127) & ~127 : 0);
  const uint32_t ring_s = smem_s + (uint32_t)(tab_bytes + xs_bytes + part_bytes);
  const uint32_t my_ring = ring_s + (uint32_t)(warp * kS * kStage);
  const uint32_t lane_base = smem_s + (uint32_t)((lane >> 4) * S) * 128u + (lane & 15) * 8u;
  uint32_t magic = 0x4B000000u;  // exponent of 2^23, kept in a register
  asm volatile("" : "+r"(magic));

  const int r0 = cta * p.rows_per_cta;
  const int nr = max(0, min(p.rows, r0 + p.rows_per_cta) - r0);
  const int nrw = warp_nrows<MODE>(warp, nr);

  // The ring starts zeroed: a lane past a ragged slice reads a stage it did
  // not fill, and must find codes in range there (its table slots are zero).
  // (2:4: position nibbles 4 = (0, 1), the smallest code the table holds)
  for (int b = 16 * lane; b < kS * kStage; b += 16 * 32) {
    const uint32_t f = N == 2 && (b % kStage) >= kIdxOff && (b % kStage) < kSzOff ? 0x44444444u : 0u;
    asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(my_ring + b), "r"(f) : "memory");
  }
  __syncwarp();
  // this lane's regions of ring stage 0 (nibbles; codes and scale/zero)
  const uint32_t ring16 = my_ring + 16 * lane, ring8 = my_ring + 8 * lane;
  RowProducer<N, MODE> prod;
  SliceCtx<N, MODE> c;
  c.prod = &prod;
  c.p = &p;
  c.ring16 = ring16;
  c.ring8 = ring8;
  c.lane_base = lane_base;
  c.magic = magic;
  c.nrw = nrw;
  c.lane = lane;

  // ---- the first two items of slice 0 into the ring (weights only: no
  // dependence on the previous kernel)
  {
    const int nch = min(p.slice_chunks, p.chunks);
    const int ipr = (nch + 31) >> 5;
    stream_prologue<N, MODE>(prod, p, r0, warp, lane, 0, ipr, nrw, lane < nch - 32 * (ipr - 1),
                             ring16, ring8);
  }

  // x of the first K slice into L2 while the previous kernel finishes: its
  // address is known now, its contents only after the wait (a prefetch
  // returns no data; a later write of x by the previous kernel lands in L2
  // all the same), so the staging below reads L2 instead of DRAM.
  if (kPrefetchX && warp == 0) {
    const int ncols = min(p.cols, p.slice_chunks * C::CPC);
    const char* xb = reinterpret_cast<const char*>(p.x);
    for (int off = 128 * lane; off < 2 * ncols; off += 128 * 32)
      asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(xb + off));
  }
  pdl_wait();
  pdl_launch_dependents();

  for (int sl = 0; sl < p.nslices; ++sl) {
    const int c0 = sl * p.slice_chunks;
    const int nch = min(p.slice_chunks, p.chunks - c0);
    const int ipr = (nch + 31) >> 5;                 // items per row
    const bool last_on = lane < nch - 32 * (ipr - 1);
    if (sl > 0)   // this warp's ring is free: the previous slice's items are consumed
      stream_prologue<N, MODE>(prod, p, r0, warp, lane, c0, ipr, nrw, last_on, ring16, ring8);
    __syncthreads();  // the previous slice's table is no longer read

    // ---- stage x of the slice (binary16, zero past cols), padded per chunk
    {
      const int ncols = nch * C::CPC;
      const int col0 = c0 * C::CPC;
      for (int t = threadIdx.x; t < ncols / 8; t += kNTm<MODE>) {
        const int col = col0 + 8 * t;
        uint4 q = make_uint4(0, 0, 0, 0);
        if (col < p.cols) q = *reinterpret_cast<const uint4*>(p.x + col);
        const int cc = (8 * t) / C::CPC, off = (8 * t) % C::CPC;
        uint32_t* dst = reinterpret_cast<uint32_t*>(xs + cc * C::XPAD + off);
        dst[0] = q.x; dst[1] = q.y; dst[2] = q.z; dst[3] = q.w;
      }
    }
    __syncthreads();

    // ---- build the pair tables: one (lane column, chunk slot, unit) per
    // thread-iteration; a warp writes 32 different lane columns at once.
    // Slots of chunks past the slice (ragged lanes) hold zeros.
    {
      const int l = threadIdx.x & 31;
      const uint32_t colbase = smem_s + (uint32_t)((l >> 4) * S) * 128u + (l & 15) * 8u;
      for (int u_it = warp; u_it < ipr * kUnitsPerChunk; u_it += kNWm<MODE>) {
        const int i = u_it / kUnitsPerChunk, u = u_it % kUnitsPerChunk;
        const int cl = l + 32 * i;
        float xv[C::UC];
        if (cl < nch) {
          const __half* src = xs + cl * C::XPAD + u * C::UC;
#pragma unroll
          for (int q = 0; q < C::UC / 2; ++q) {
            const __half2 h2 = *reinterpret_cast<const __half2*>(src + 2 * q);
            xv[2 * q] = __low2float(h2);
            xv[2 * q + 1] = __high2float(h2);
          }
        } else {
#pragma unroll
          for (int q = 0; q < C::UC; ++q) xv[q] = 0.0f;
        }
        const uint32_t a = colbase + (uint32_t)(i * C::SLOTS + u * C::E) * 128u;
        if constexpr (N == 2) {
#pragma unroll
          for (int e = 0; e < 6; ++e) {
            const int nib = quad24_nibble(e);
            sts_pair(a + (nib - 4) * 128, xv[nib & 3], xv[nib >> 2]);
          }
        } else {
#pragma unroll
          for (int e = 0; e < C::E; ++e) sts_pair(a + e * 128, xv[e & 3], xv[4 + (e >> 2)]);
        }
      }
    }
    __syncthreads();

    // ---- stream the warp's rows of this slice
    c.c0 = c0;
    c.last_on = last_on;
    c.par = 0;
    switch (ipr) {
      case 1: stream_slice<N, MODE, 1>(c, r0, warp, sl, part); break;
      case 2: stream_slice<N, MODE, 2>(c, r0, warp, sl, part); break;
      case 3: if constexpr (max_ipr<N>() >= 3) stream_slice<N, MODE, 3>(c, r0, warp, sl, part); break;
      case 4: if constexpr (max_ipr<N>() >= 4) stream_slice<N, MODE, 4>(c, r0, warp, sl, part); break;
      default: break;   // the plan never makes more
    }
  }
  cp_wait<0>();  // no copy outstanding when the CTA retires
}

template <int N, int MODE>
__global__ void __launch_bounds__(kNTm<MODE>, 1) k_m1(const __grid_constant__ M1Params p) {
  m1_body<N, MODE>(p, blockIdx.x);
}

// Matrices of both N that share x in one launch: CTAs [0, grid_a) run the
// 2:4 part, the others the 1:4 part; each builds only its own pair table.
struct M1DualParams {
  M1Params a, b;
  int grid_a;
};

__global__ void __launch_bounds__(kNTm<kMany>, 1) k_m1_dual(const __grid_constant__ M1DualParams p) {
  if ((int)blockIdx.x < p.grid_a)
    m1_body<2, kMany>(p.a, blockIdx.x);
  else
    m1_body<1, kMany>(p.b, blockIdx.x - p.grid_a);
}

// Time of a 1:4 chunk against a 2:4 chunk in the M=1 kernel (a CTA-time
// trace of the mixed q/k/v launch; 1.3 gave the shortest step of 1.0-1.5)
#ifndef SGEMV_M1_PDL
#define SGEMV_M1_PDL 1
#endif
#ifndef SGEMV_M1_COST14
#define SGEMV_M1_COST14 1.3
#endif
constexpr double kCost14 = SGEMV_M1_COST14;

int g_num_sms[64] = {0};

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev < 0 || dev >= 64) return 0;
  if (!g_num_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return 0;
    g_num_sms[dev] = n;
  }
  return g_num_sms[dev];
}

// The plan of one launch part over `count` matrices that share x, cols and
// N (count <= kMaxSeg), for `ctas` CTAs: parameters, grid and shared memory.
template <int N, int MODE>
cudaError_t plan_m1(const Layout* Ls, const RunArgs* as, int count, int ctas, M1Params& p,
                    int& grid, size_t& smem) {
  using C = M1Cfg<N>;
  const Layout& L0 = Ls[0];
  const int chunks = (int)L0.chunks;
  int64_t total_rows = 0;
  for (int i = 0; i < count; ++i) {
    if ((int64_t)Ls[i].rows * Ls[i].cstride >= (1ll << 31) ||
        (int64_t)Ls[i].rows * Ls[i].gstride >= (1ll << 31))
      return cudaErrorNotSupported;
    total_rows += Ls[i].rows;
  }
  grid = 0;
  smem = 0;
  if (total_rows == 0) return cudaSuccess;
  if (total_rows >= (1ll << 31)) return cudaErrorNotSupported;
  if (ctas <= 0) return cudaErrorNotSupported;
  const size_t ring = (size_t)kNWm<MODE> * kS * kStage;
  const size_t part_max = 4096;   // rows_per_cta <= 1024 when K is sliced
  const size_t room = kSmemLimit - kTabAlign - ring - part_max;
  const int max_cpl = min((int)(room / (C::TAB_PER_CPL + C::X_PER_CPL)), max_ipr<N>());
  if (max_cpl < 1) return cudaErrorNotSupported;
  const int nslices = (chunks + 32 * max_cpl - 1) / (32 * max_cpl);
  const int cpl = (chunks + 32 * nslices - 1) / (32 * nslices);
  const int rows = (int)total_rows;
  int rows_per_cta = (rows + ctas - 1) / ctas;
  if (nslices > 1 && rows_per_cta > 1024) rows_per_cta = 1024;
  grid = (rows + rows_per_cta - 1) / rows_per_cta;

  memset(&p, 0, sizeof p);
  int row_begin = 0;
  for (int i = 0; i < count; ++i) {
    M1Seg& sg = p.seg[i];
    sg.vals = as[i].vals;
    sg.idx = as[i].idx;
    sg.sz = as[i].sz;
    sg.y = as[i].y;
    sg.row_begin = row_begin;
    sg.gstride = (int)Ls[i].gstride;
    sg.gshift = Ls[i].group == 64 ? 6 : (Ls[i].group == 128 ? 7 : 8);
    sg.g64 = N == 1 && Ls[i].group == 64;
    row_begin += Ls[i].rows;
  }
  // empty matrices may sit anywhere in the list; unused entries start past
  // the row space so the lookup never selects them
  for (int i = count; i < kMaxSeg; ++i) p.seg[i].row_begin = rows;
  p.nseg = count;
  p.x = as[0].x;
  p.err = as[0].err;
  p.rows = rows;
  p.cols = L0.cols;
  p.cstride = (int)L0.cstride;
  p.chunks = chunks;
  p.rows_per_cta = rows_per_cta;
  p.cpl = cpl;
  p.slice_chunks = 32 * cpl;
  p.nslices = nslices;

  const size_t part_bytes = nslices > 1 ? ((size_t)rows_per_cta * 4 + 127) & ~(size_t)127 : 0;
  smem = kTabAlign + (size_t)cpl * (C::TAB_PER_CPL + C::X_PER_CPL) + part_bytes + ring;
  if (smem > (size_t)kSmemLimit) return cudaErrorNotSupported;
  return cudaSuccess;
}

template <typename Kernel, typename Params>
cudaError_t launch_pdl(Kernel kernel, const Params& p, int grid, int threads, size_t smem,
                       cudaStream_t s, bool (&attr_set)[64]) {
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemLimit);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = SGEMV_M1_PDL ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

// One launch over `count` matrices that share x, cols and N (count <= kMaxSeg).
template <int N, int MODE>
cudaError_t launch_m1_n(const Layout* Ls, const RunArgs* as, int count, cudaStream_t s) {
  M1Params p;
  int grid;
  size_t smem;
  cudaError_t e = plan_m1<N, MODE>(Ls, as, count, num_sms(), p, grid, smem);
  if (e != cudaSuccess || grid == 0) return e;
  static bool attr_set[64] = {false};
  return launch_pdl(k_m1<N, MODE>, p, grid, kNTm<MODE>, smem, s, attr_set);
}

}  // namespace

cudaError_t launch_m1(const Layout& L, const RunArgs& a, cudaStream_t s) {
  if (a.m != 1 || L.rows == 0 || L.cols == 0) return cudaErrorNotSupported;
  if (L.n_keep == 2) return launch_m1_n<2, kOne>(&L, &a, 1, s);
  return L.group == 64 ? launch_m1_n<1, kOneG64>(&L, &a, 1, s)
                       : launch_m1_n<1, kOne>(&L, &a, 1, s);
}

cudaError_t launch_m1_group(const Layout* Ls, const RunArgs* as, int count, cudaStream_t s) {
  if (count < 1 || count > kMaxSeg) return cudaErrorNotSupported;
  for (int i = 0; i < count; ++i)
    if (as[i].m != 1 || Ls[i].cols != Ls[0].cols || Ls[i].n_keep != Ls[0].n_keep ||
        Ls[i].cols == 0)
      return cudaErrorNotSupported;
  return Ls[0].n_keep == 2 ? launch_m1_n<2, kMany>(Ls, as, count, s)
                           : launch_m1_n<1, kMany>(Ls, as, count, s);
}

cudaError_t launch_m1_group_dual(const Layout* L2, const RunArgs* a2, int n2, const Layout* L1,
                                 const RunArgs* a1, int n1, cudaStream_t s) {
  if (n2 < 1 || n2 > kMaxSeg || n1 < 1 || n1 > kMaxSeg) return cudaErrorNotSupported;
  for (int i = 0; i < n2; ++i)
    if (a2[i].m != 1 || L2[i].cols != L2[0].cols || L2[i].n_keep != 2 || L2[i].cols == 0)
      return cudaErrorNotSupported;
  for (int i = 0; i < n1; ++i)
    if (a1[i].m != 1 || L1[i].cols != L2[0].cols || L1[i].n_keep != 1)
      return cudaErrorNotSupported;
  const int sms = num_sms();
  if (sms < 2) return cudaErrorNotSupported;
  // CTAs in proportion to each part's time: its chunks (32 kept weights
  // each) times the measured cost of a chunk, kCost14 for 1:4 (larger pair
  // tables and units of two quads) against 1 for 2:4
  double b2 = 0.0, b1 = 0.0;
  for (int i = 0; i < n2; ++i) b2 += (double)L2[i].rows * L2[i].chunks;
  for (int i = 0; i < n1; ++i) b1 += kCost14 * L1[i].rows * L1[i].chunks;
  if (b2 <= 0.0 || b1 <= 0.0) return cudaErrorNotSupported;
  int c2 = (int)(sms * b2 / (b1 + b2) + 0.5);
  c2 = c2 < 1 ? 1 : (c2 > sms - 1 ? sms - 1 : c2);
  M1DualParams p;
  int g2, g1;
  size_t s2, s1;
  cudaError_t e = plan_m1<2, kMany>(L2, a2, n2, c2, p.a, g2, s2);
  if (e != cudaSuccess) return e;
  e = plan_m1<1, kMany>(L1, a1, n1, sms - c2, p.b, g1, s1);
  if (e != cudaSuccess) return e;
  if (g2 == 0 || g1 == 0) return cudaErrorNotSupported;
  p.grid_a = g2;
  static bool attr_set[64] = {false};
  return launch_pdl(k_m1_dual, p, g2 + g1, kNTm<kMany>, s2 > s1 ? s2 : s1, s, attr_set);
}

int max_group() { return kMaxSeg; }

}  // namespace sgemv
