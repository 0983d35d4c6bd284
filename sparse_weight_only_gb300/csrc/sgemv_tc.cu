// sgemv_tc.cu -- SparseGemv for a batch of activation rows (2 <= m <= 64:
// beam candidates / prefix-tree verification nodes) on the fifth-generation
// tensor cores: tcgen05.mma.sp with the accumulators in tensor memory.
//
// Product (Dong et al., arXiv 2605.11582, section 1 contribution 2 and
// section 3.3, applied to the verification batch of section 3.1):
//   y[m][r] = sum_G s_rG * sum_{kept j in G} (q_j - z_rG) * x[m][col_j],
// each product exact, fp32 accumulation, one binary16 rounding per output.
//
// The weight is the MMA's A operand (M = 128 weight rows per tile), x the B
// operand (N = m rounded up to 16), and the 2:4 sparse MMA consumes the
// stored in-quad positions directly as its metadata:
//  * A: each thread owns one weight row (= one tensor-memory lane) and
//    decodes its kept weights to exact binary16 (q - z) -- PRMT + LOP3 +
//    HSUB2 per quad, an integer in [-15, 15] -- then writes them to tensor
//    memory with tcgen05.st; one tensor-memory column holds one quad's two
//    kept values.  1:4 weights pair each kept value with a zero at the other
//    position of its half of the quad, so the 2:4 MMA computes exactly its
//    product.
//  * metadata: the 2:4 position nibbles a | b << 2 of a row's eight quads of
//    a 32-column k-step are one 32-bit word; tensor memory holds them as the
//    warp-level sparse MMA does in registers -- within each 16 rows, lane i
//    (i < 8) carries quads 0..3 of rows i and i + 8, lane i + 8 quads 4..7
//    -- so each row thread exchanges half of its word with lane ^ 8.
//  * B: x arrives by TMA in 128-byte-swizzled K-major tiles, 64 columns per
//    tile, one shared-memory descriptor per 32-column k-step.
//  * scale: every quantisation group's k-steps accumulate into a tensor-memory
//    block of their own; the row threads load it (tcgen05.ld), multiply by
//    the group's fp32 scale and add into fp32 registers.
//  * weights: a unit of 4 chunks (256 columns at 2:4, 512 at 1:4) of 128 rows
//    comes in by three TMA tile loads (positions, codes, scale/zero words)
//    into a ring of shared-memory stages filled well ahead of use.
//  * work split: a persistent grid of one CTA per SM takes equal runs of the
//    (row tile, K unit) sequence.  A tile whose units span several CTAs is
//    finished by the last of them to arrive: each writes its fp32 partial to
//    the handle's split-K workspace and bumps the tile's counter; the last
//    sums the partials in CTA order (deterministic) and writes y.  No CTA
//    ever waits for another.
//  * every wait on an mbarrier is bounded; one that runs out records
//    SGEMV_ERR_TIMEOUT, the CTA stops issuing work, lets the copies it
//    issued land and frees its tensor memory.
#include <cuda.h>
#include <string.h>

#include "sgemv_internal.cuh"

namespace sgemv {
namespace {

constexpr int kThreads = 480;          // 15 warps: 8 decode, 4 epilogue, 2 MMA issue, TMA producer
constexpr int kRows = 128;             // weight rows per tile (MMA M)
constexpr int kNW = 6;                 // weight units in the shared-memory ring
constexpr int kNX = 6;                 // x sub-stages in the ring (refilled 2 behind)
constexpr int kTmemCols = 512;
// one weight unit: codes 128 rows x 64 B (64-byte swizzle) | positions
// 128 x 32 B (32-byte swizzle) | scale/zero words 128 x 32 B
constexpr int kStageW = 16384;
constexpr int kValsOff = 0, kIdxOff = 8192, kSzOff = 12288;
constexpr int kSzWords = 8;            // scale/zero words per row and unit
constexpr unsigned long long kWaitLimitNs = 1000000000ull;
constexpr unsigned long long kInjectWaitNs = 20000ull;

// One packed matrix of a launch: a launch covers up to kTcMaxSeg matrices
// that share x, cols, N and the group size; their 128-row tiles are
// numbered in order.
constexpr int kTcMaxSeg = 4;
struct TcSeg {
  CUtensorMap tm_vals, tm_idx, tm_sz;
  __half* y;
  int* counters;         // [this matrix's tiles] arrivals per tile (left at 0)
  int rows;
  int tile_begin;        // first tile of this matrix in the launch
};

struct TcParams {
  TcSeg seg[kTcMaxSeg];
  CUtensorMap tm_x;
  float* scratch;        // [grid][2][128][npad] fp32 partial tiles
  int* err;
  int nseg;
  int cols, m;
  int group, gshift;
  int ntiles, units_per_tile;
  long long total_units;
  int grid;
  int parts;             // >= 2: each tile's units split over a cluster of `parts` CTAs
                         // (split-K through distributed shared memory); else stream-K
  int withhold;          // failure-detection test hook: no x loads are issued
  unsigned long long wait_ns;
};

// ---- PTX helpers -----------------------------------------------------------
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Non-blocking test (try_wait may suspend the thread for a while): for a
// thread that polls several barriers in turn.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void tma_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                       uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Thread-block cluster: a full barrier (release / acquire), the address of
// the same shared-memory offset in another CTA of the cluster, and a 16-byte
// load from there.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t mapa_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
// 128-byte-swizzled K-major shared-memory operand (8-row atoms, 1024 B apart)
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFF) >> 4) | (1ull << 16) | ((uint64_t)(1024 >> 4) << 32) |
         (1ull << 46) | (2ull << 61);
}
__device__ __forceinline__ void mma_sp(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t meta,
                                       uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %5, 0;\n"
      " tcgen05.mma.sp.cta_group::1.kind::f16 [%0], [%1], %2, [%3], %4, p;\n}" ::"r"(d),
      "r"(a), "l"(bdesc), "r"(meta), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   bar)
               : "memory");
}
__device__ __forceinline__ void st8(uint32_t taddr, const uint32_t (&v)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
               "r"(v[7])
               : "memory");
}
__device__ __forceinline__ void st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
__device__ __forceinline__ void ld8(uint32_t taddr, uint32_t (&v)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]),
                 "=r"(v[6]), "=r"(v[7])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}

// ---- decode ---------------------------------------------------------------
// (1024 + z, 64 + z) as half2 from a scale/zero word (zero in the high half)
__device__ __forceinline__ uint32_t zconst(uint32_t szw) {
  const uint32_t zz = __byte_perm(szw, 0u, 0x3232u);
  uint32_t zc;
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(zc) : "r"(zz), "r"(0x54006400u));
  return zc;
}
// 2:4: half2 (q_a - z, q_b - z) of the quad in byte `b` of w: the byte goes to
// bytes 0 and 2, its low nibble into the mantissa of 1024, its high nibble
// into that of 64, and one subtraction removes (1024 + z, 64 + z).
__device__ __forceinline__ uint32_t quad24(uint32_t w, int b, uint32_t zc) {
  uint32_t t = __byte_perm(w, 0u, 0x4040u | (uint32_t)b | ((uint32_t)b << 8));
  asm("lop3.b32 %0, %1, 0x00F0000F, 0x54006400, 0xEA;" : "=r"(t) : "r"(t));
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(t), "r"(zc));
  return d;
}
// 1:4: the A words of quads c and c + 4 (c < 4) of a k-step: the nibbles of
// word w (one per quad) decode pairwise, and each value goes to the low half
// (even position) or high half (odd position) of its word, the other half 0.
__device__ __forceinline__ void quads14(uint32_t w, int c, uint32_t pos, uint32_t z1024,
                                        uint32_t& a_c, uint32_t& a_c4) {
  uint32_t t;
  asm("lop3.b32 %0, %1, 0x000F000F, 0x64006400, 0xEA;" : "=r"(t) : "r"(w >> (4 * c)));
  uint32_t v;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(v) : "r"(t), "r"(z1024));   // (v_c, v_c4)
  const uint32_t odd_c = (pos >> (2 * c)) & 1u, odd_c4 = (pos >> (2 * c + 8)) & 1u;
  a_c = __byte_perm(v, 0u, 0x4410u - odd_c * 0x33CCu);    // (v,0) or (0,v)
  a_c4 = __byte_perm(v, 0u, 0x4432u - odd_c4 * 0x11EEu);
}
// 1:4 metadata word of a k-step from its 16 position bits (quad c at bits
// 2c): nibble c is 4 = (0, 1) when the position is 0 or 1, else 14 = (2, 3).
__device__ __forceinline__ uint32_t meta14(uint32_t pos16) {
  uint32_t x = (pos16 >> 1) & 0x5555u;            // high bit of quad c at bit 2c
  x = (x | (x << 8)) & 0x00FF00FFu;
  x = (x | (x << 4)) & 0x0F0F0F0Fu;
  x = (x | (x << 2)) & 0x33333333u;
  x = (x | (x << 1)) & 0x55555555u;               // ... at bit 4c
  return 0x44444444u | (x * 10u);
}
// The tensor-memory lane word of a row's metadata word (lane ^ 8 exchange).
__device__ __forceinline__ uint32_t meta_lane(uint32_t mw, int lane) {
  const uint32_t p = __shfl_xor_sync(0xffffffffu, mw, 8);
  return (lane & 8) ? __byte_perm(p, mw, 0x7632u) : __byte_perm(mw, p, 0x5410u);
}

// ---- the kernel -----------------------------------------------------------
// Sequence of the CTA's work: units u in [u_begin, u_end) of the linear
// (tile, unit) order; each unit is SUBS sub-stages of four 32-column
// k-steps.  A "segment" is the CTA's run of units inside one tile; a group
// "instance" is a maximal run of the segment's k-steps inside one
// quantisation group inside one sub-stage and owns one accumulator block.
// Every role walks the same sequence; they meet only at mbarriers:
//   producer (warp 14)  --weights-->  decode warps 0-7  --A, metadata-->
//   MMA warps 12, 13  --accumulator blocks-->  epilogue warps 8-11  --y
// Weight units have a full and an empty barrier, x sub-stages and A slots a
// full one; a single MMA commit per sub-stage ("sub-stage done") frees its
// A slot and x slot and finalises its accumulator blocks; the epilogue
// frees each block for reuse.

// The walk over the CTA's units: position (tile, unit in tile) stepped
// forward in 32-bit arithmetic, and the segment bounds.
struct Walk {
  int U, nunits;
  int tile, uit, seg_u0;
  __device__ __forceinline__ Walk(int U_, int nunits_, int tile0, int uit0)
      : U(U_), nunits(nunits_), tile(tile0), uit(uit0), seg_u0(uit0) {}
  // call at the first sub-stage of unit ui > 0
  __device__ __forceinline__ void next_unit() {
    if (++uit == U) {
      uit = 0;
      ++tile;
      seg_u0 = 0;
    }
  }
  __device__ __forceinline__ int seg_u1(int ui) const { return min(U, uit + (nunits - ui)); }
  __device__ __forceinline__ bool unit_ends_segment(int ui) const {
    return ui + 1 == nunits || uit + 1 == U;
  }
};

// The workspace slot in which the first CTA sharing a tile (c0, whose range
// starts at unit b0) wrote it: slot 0 holds a CTA's first split segment,
// and the tile is c0's first one when c0 starts inside it or on a tile
// boundary (a whole first tile goes to y directly); otherwise slot 1.
// Every later CTA sharing the tile starts inside it: slot 0.
__device__ __forceinline__ int split_slot0(int c0, long long tu0, long long T, int P, int U) {
  const long long b0 = (long long)c0 * T / P;
  return b0 >= tu0 || b0 % U == 0 ? 0 : 1;
}

// The k-steps of one sub-stage: which are inside K, which start and end a
// group instance, and the instance each belongs to.  An instance never
// spans two sub-stages (a 256-column group is two instances, each scaled
// by the group's scale), so every sub-stage's MMAs stand alone.
struct Steps {
  int ij[4];
  bool valid[4], first[4], ends[4];
  __device__ __forceinline__ void walk(int scol0, int seg_c1, int group, int& inst) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int col = scol0 + 32 * j;
      valid[j] = col < seg_c1;
      first[j] = false;
      ends[j] = false;
      if (valid[j]) {
        if (j == 0 || (col & (group - 1)) == 0) {
          ++inst;
          first[j] = true;
        }
        ends[j] = j == 3 || col + 32 >= seg_c1 || ((col + 32) & (group - 1)) == 0;
      }
      ij[j] = inst;
    }
  }
};

constexpr int kDecodeWarps = 8;
constexpr int kEpiWarp0 = 8;           // epilogue warps 8..11 (lane quadrant w - 8)
constexpr int kMmaWarp = 12;           // MMA issue: warps 12 and 13, alternate sub-stages
constexpr int kProdWarp = 14;
constexpr int kRD = 32;                // "sub-stage done" barriers (ring)
#ifndef SGEMV_TC_ALIGN_PCT
#define SGEMV_TC_ALIGN_PCT 50
#endif
constexpr int kAlignPct = SGEMV_TC_ALIGN_PCT;   // least share of the SMs a tile-aligned grid keeps
#ifndef SGEMV_TC_DEC2
#define SGEMV_TC_DEC2 1
#endif
// Decode warps take sub-stages in pairs: both decodes before both stores,
// so that the two dependency chains interleave (1.5% off the config-4
// verification step at M = 17..64).
constexpr bool kDecodePairs = SGEMV_TC_DEC2 != 0;
#ifndef SGEMV_TC_CLUSTER
#define SGEMV_TC_CLUSTER 1
#endif
constexpr bool kClusterMode = SGEMV_TC_CLUSTER != 0;

// The matrix of launch tile `tile`.
__device__ __forceinline__ const TcSeg& seg_of(const TcParams& p, int tile) {
  int s = 0;
  while (s + 1 < p.nseg && tile >= p.seg[s + 1].tile_begin) ++s;
  return p.seg[s];
}
// Row r of launch tile `tile` in its matrix's y (m x rows, row-major).
struct YRow {
  __half* y;
  int rows, row;
  __device__ __forceinline__ YRow(const TcParams& p, int tile, int r) {
    const TcSeg& sg = seg_of(p, tile);
    y = sg.y;
    rows = sg.rows;
    row = (tile - sg.tile_begin) * kRows + r;
  }
  __device__ __forceinline__ bool valid() const { return row < rows; }
  __device__ __forceinline__ void put(int i, int m, float v) const {
    if (i < m && row < rows) y[(size_t)i * rows + row] = __float2half_rn(v);
  }
};

template <int N, int NPAD>
__global__ void __launch_bounds__(kThreads, 1) k_tc(const __grid_constant__ TcParams p) {
  constexpr int SUBS = N == 2 ? 2 : 4;           // sub-stages per unit
  constexpr int UNIT_COLS = 128 * SUBS;          // 256 or 512 dense columns
  constexpr int XBOX = NPAD * 128;               // bytes of one 64-column x tile
  constexpr int XSUB = 2 * XBOX;
  constexpr int DCOLS = NPAD <= 32 ? 128 : 256;  // accumulator region of tensor memory
  constexpr int ND = DCOLS / NPAD;               // accumulator blocks
  constexpr int NA = (kTmemCols - DCOLS) / 128;  // A/metadata slots (sub-stages)
  constexpr uint32_t IDESC = (1u << 2) | (1u << 4) | ((uint32_t)(NPAD >> 3) << 17) |
                             ((uint32_t)(kRows >> 4) << 24);

  extern __shared__ __align__(1024) unsigned char smem_raw[];
  const uint32_t raw = (uint32_t)__cvta_generic_to_shared(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* sm = smem_raw + (base - raw);
  const uint32_t wring = base;
  const uint32_t xring = base + kNW * kStageW;
  const uint32_t bars = xring + kNX * XSUB;
  // weight unit full / empty; x sub-stage full; A/metadata slot full; the
  // "sub-stage done" ring (one MMA commit per sub-stage: its A slot, x slot
  // and accumulator blocks are then free / final); accumulator block empty
  const uint32_t bar_wf = bars, bar_we = bar_wf + 8 * kNW;
  const uint32_t bar_xf = bar_we + 8 * kNW;
  const uint32_t bar_af = bar_xf + 8 * kNX;
  const uint32_t bar_dn = bar_af + 8 * NA;
  const uint32_t bar_de = bar_dn + 8 * kRD;
  const uint32_t misc = bar_de + 8 * ND;
  volatile uint32_t* tmem_slot = reinterpret_cast<volatile uint32_t*>(sm + (misc - base));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + (misc - base) + 4);
  volatile int* last_flag = reinterpret_cast<volatile int*>(sm + (misc - base) + 8);
  volatile int* pub = reinterpret_cast<volatile int*>(sm + (misc - base) + 12);  // w, x, mma ends
  // the tile whose split-K sum this CTA does after its teardown barrier, or -1
  volatile int* final_tile = reinterpret_cast<volatile int*>(sm + (misc - base) + 32);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  const int U = p.units_per_tile;
  const long long T = p.total_units;
  const int P = p.grid;
  // the CTA's run of (row tile, K unit) units: equal runs of the whole
  // sequence (stream-K), or -- in cluster mode -- part (rank) q of tile t
  long long u_begin, u_end;
  if (p.parts >= 2) {
    const int t = (int)blockIdx.x / p.parts, q = (int)blockIdx.x % p.parts;
    u_begin = (long long)t * U + (long long)q * U / p.parts;
    u_end = (long long)t * U + (long long)(q + 1) * U / p.parts;
  } else {
    u_begin = (long long)blockIdx.x * T / P;
    u_end = (long long)(blockIdx.x + 1) * T / P;
  }
  const int nunits = (int)(u_end - u_begin);
  const int nsub = nunits * SUBS;
  const int tile0 = (int)(u_begin / U), uit0 = (int)(u_begin % U);

  if (tid == 0) {
    for (int i = 0; i < kNW; ++i) {
      mbar_init(bar_wf + 8 * i, 1);
      mbar_init(bar_we + 8 * i, kDecodeWarps + 4);
    }
    for (int i = 0; i < kNX; ++i) mbar_init(bar_xf + 8 * i, 1);
    for (int i = 0; i < NA; ++i) mbar_init(bar_af + 8 * i, kDecodeWarps);
    for (int i = 0; i < kRD; ++i) mbar_init(bar_dn + 8 * i, 1);
    for (int i = 0; i < ND; ++i) mbar_init(bar_de + 8 * i, 4);
    *abort_flag = 0;
    *final_tile = -1;
    pub[0] = pub[1] = pub[2] = pub[3] = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(misc),
                 "n"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *tmem_slot;

  // bounded wait: false when it ran out (then abort is set) or another role aborted
  auto wait = [&](uint32_t bar, uint32_t parity) -> bool {
    if (mbar_try(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try(bar, parity)) {
      if (*abort_flag) return false;
      if (global_ns() - t0 > p.wait_ns) {
        *abort_flag = 1;
        atomicCAS(p.err, 0, kDevErrTimeout);
        return false;
      }
    }
    return true;
  };

  if (warp == kProdWarp) {
    // ======================= producer: TMA copies =========================
    if (lane == 0) {
      int w_issued = 0, x_issued = 0;
      int w_tile = tile0, w_uit = uit0, x_uit = uit0, x_ls = 0;
      auto issue_w = [&]() {
        const uint32_t dst = wring + (uint32_t)((w_issued % kNW) * kStageW);
        const uint32_t bar = bar_wf + 8 * (w_issued % kNW);
        mbar_expect_tx(bar, kStageW);
        const int chunk0 = w_uit * 4;
        const int g0 = ((w_uit * UNIT_COLS) >> p.gshift) & ~3;
        const TcSeg& sg = seg_of(p, w_tile);
        const int wrow = (w_tile - sg.tile_begin) * kRows;
        tma_2d(dst + kValsOff, &sg.tm_vals, chunk0 * 16, wrow, bar);
        tma_2d(dst + kIdxOff, &sg.tm_idx, chunk0 * 8, wrow, bar);
        tma_2d(dst + kSzOff, &sg.tm_sz, g0, wrow, bar);
        ++w_issued;
        if (++w_uit == U) {
          w_uit = 0;
          ++w_tile;
        }
      };
      auto issue_x = [&]() {
        const int col0 = x_uit * UNIT_COLS + x_ls * 128;
        const uint32_t dst = xring + (uint32_t)((x_issued % kNX) * XSUB);
        const uint32_t bar = bar_xf + 8 * (x_issued % kNX);
        mbar_expect_tx(bar, XSUB);
        tma_2d(dst, &p.tm_x, col0, 0, bar);
        tma_2d(dst + XBOX, &p.tm_x, col0 + 64, 0, bar);
        ++x_issued;
        if (++x_ls == SUBS) {
          x_ls = 0;
          if (++x_uit == U) x_uit = 0;
        }
      };
      // the weights do not depend on the previous kernel: in flight before the wait
      while (w_issued < min(nunits, kNW)) issue_w();
      asm volatile("griddepcontrol.wait;" ::: "memory");
      const int x_total = p.withhold ? 0 : nsub;
      unsigned long long t0 = global_ns();
      while ((w_issued < nunits || x_issued < x_total) && !*abort_flag) {
        bool moved = false;
        if (x_issued < x_total &&
            (x_issued < kNX || mbar_test(bar_dn + 8 * ((x_issued - kNX) % kRD),
                                         (uint32_t)(((x_issued - kNX) / kRD) & 1)))) {
          issue_x();
          moved = true;
        }
        if (w_issued < nunits &&
            mbar_test(bar_we + 8 * (w_issued % kNW), (uint32_t)(((w_issued / kNW) - 1) & 1))) {
          issue_w();
          moved = true;
        }
        if (moved) {
          t0 = global_ns();
        } else if (global_ns() - t0 > p.wait_ns) {
          *abort_flag = 1;
          atomicCAS(p.err, 0, kDevErrTimeout);
        }
      }
      pub[0] = w_issued;
      pub[1] = x_issued;
    }
  } else {
    asm volatile("griddepcontrol.wait;" ::: "memory");
  }
  asm volatile("griddepcontrol.launch_dependents;");

  if (warp < kDecodeWarps) {
    // ======================= decode: weights -> A, metadata ===============
    const int quad = warp & 3, h = warp >> 2;
    const int r = quad * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    int uit = uit0, dtile = tile0;   // dtile: read by the checked build only
    // sub-stage s of the weights -> A and metadata registers (false: a wait
    // gave up)
    auto decode_sub = [&](int s, uint32_t (&a0)[8], uint32_t (&a1)[8], uint32_t& m0,
                          uint32_t& m1) -> bool {
      const int ui = s / SUBS, ls = s % SUBS;
      if (ls == 0 && ui > 0 && ++uit == U) {
        uit = 0;
        ++dtile;
      }
      const uint32_t wslot = wring + (uint32_t)((ui % kNW) * kStageW);
      if (ls == 0 && !__all_sync(0xffffffffu, wait(bar_wf + 8 * (ui % kNW), (uint32_t)((ui / kNW) & 1))))
        return false;
      const int scol0 = uit * UNIT_COLS + ls * 128;
      const int g0 = ((uit * UNIT_COLS) >> p.gshift) & ~3;
      int myG = (scol0 + 64 * h) >> p.gshift;
      if constexpr (kChecked) {
        if (myG - g0 < 0 || myG - g0 >= kSzWords) {
          report_checked(p.err);
          myG = g0;
        }
      }
      const uint32_t szw = lds32(wslot + kSzOff + (uint32_t)(r * 32 + (myG - g0) * 4));
      if constexpr (N == 2) {
        const int ch = 2 * ls + h;
        const uint4 v = lds128(wslot + kValsOff + (uint32_t)(r * 64 + ((ch ^ ((r >> 1) & 3)) << 4)));
        const uint2 ix = lds64(wslot + kIdxOff +
                               (uint32_t)(r * 32 + ((ls ^ ((r >> 2) & 1)) << 4) + h * 8));
        const uint32_t zc = zconst(szw);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          a0[c] = quad24(c < 4 ? v.x : v.y, c & 3, zc);
          a1[c] = quad24(c < 4 ? v.z : v.w, c & 3, zc);
        }
        m0 = ix.x;
        m1 = ix.y;
        if constexpr (kChecked) {
          // valid rows and columns only: the zero padding past the matrix
          // (rows of the last tile, columns past K) is never multiplied
          const int colv = uit * UNIT_COLS + ls * 128 + 64 * h;
          const bool rowv = YRow(p, dtile, r).valid();
          if (rowv && ((colv < p.cols && bad_codes24(m0)) || (colv + 32 < p.cols && bad_codes24(m1)))) {
            report_checked(p.err);
            m0 = m1 = 0x44444444u;
          }
        }
      } else {
        const uint2 v = lds64(wslot + kValsOff +
                              (uint32_t)(r * 64 + ((ls ^ ((r >> 1) & 3)) << 4) + h * 8));
        const uint32_t pw = lds32(wslot + kIdxOff +
                                  (uint32_t)(r * 32 + (((ls >> 1) ^ ((r >> 2) & 1)) << 4) +
                                             (ls & 1) * 8 + h * 4));
        const uint32_t z1024 = __byte_perm(zconst(szw), 0u, 0x1010u);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          quads14(v.x, c, pw, z1024, a0[c], a0[c + 4]);
          quads14(v.y, c, pw >> 16, z1024, a1[c], a1[c + 4]);
        }
        m0 = meta14(pw & 0xFFFFu);
        m1 = meta14(pw >> 16);
      }
      m0 = meta_lane(m0, lane);
      m1 = meta_lane(m1, lane);
      if (ls == SUBS - 1) {   // this warp is done with the unit's shared memory
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_we + 8 * (ui % kNW));
      }
      return true;
    };
    // ... -> tensor memory, once the A/metadata slot is free
    auto store_sub = [&](int s, const uint32_t (&a0)[8], const uint32_t (&a1)[8], uint32_t m0,
                         uint32_t m1) -> bool {
      // the A/metadata slot of s is free once the MMAs of s - NA are done
      const int t = s % NA;
      if (s >= NA && !__all_sync(0xffffffffu, wait(bar_dn + 8 * ((s - NA) % kRD),
                                                    (uint32_t)(((s - NA) / kRD) & 1))))
        return false;
      fence_after();
      const uint32_t slot_col = (uint32_t)(DCOLS + 32 * (4 * t + 2 * h));
      st8(tmem + lane_off + slot_col + 8, a0);
      st8(tmem + lane_off + slot_col + 32 + 8, a1);
      st1(tmem + lane_off + slot_col, m0);
      st1(tmem + lane_off + slot_col + 32, m1);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_af + 8 * t);
      return true;
    };
    if (kDecodePairs) {
      // two sub-stages per pass: their decodes interleave, and the loop and
      // waits are paid once per pair
      for (int s = 0; s < nsub; s += 2) {
        uint32_t a0[8], a1[8], b0[8], b1[8], m0, m1, n0, n1;
        const bool two = s + 1 < nsub;
        if (!decode_sub(s, a0, a1, m0, m1)) break;
        if (two && !decode_sub(s + 1, b0, b1, n0, n1)) break;
        if (!store_sub(s, a0, a1, m0, m1)) break;
        if (two && !store_sub(s + 1, b0, b1, n0, n1)) break;
      }
    } else {
      for (int s = 0; s < nsub; ++s) {
        uint32_t a0[8], a1[8], m0, m1;
        if (!decode_sub(s, a0, a1, m0, m1)) break;
        if (!store_sub(s, a0, a1, m0, m1)) break;
      }
    }
  } else if (warp == kMmaWarp || warp == kMmaWarp + 1) {
    // ======================= MMA issue ====================================
    // Two threads in two warps take alternate sub-stages (a sub-stage's MMAs
    // stand alone: its own A slot, x slot and accumulator blocks).
    if (lane == 0) {
      const int mine = warp - kMmaWarp;
      Walk wk(U, nunits, tile0, uit0);
      int inst = -1, s_end = 0;
      for (int s = 0; s < nsub && !*abort_flag; ++s) {
        const int ui = s / SUBS, ls = s % SUBS;
        if (ls == 0 && ui > 0) wk.next_unit();
        const int seg_c1 = min(p.cols, wk.seg_u1(ui) * UNIT_COLS);
        Steps st;
        st.walk(wk.uit * UNIT_COLS + ls * 128, seg_c1, p.group, inst);
        if ((s & 1) != mine) continue;
        const int t = s % NA;
        if (!wait(bar_af + 8 * t, (uint32_t)((s / NA) & 1))) break;
        if (!wait(bar_xf + 8 * (s % kNX), (uint32_t)((s / kNX) & 1))) break;
        bool ok = true;
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (st.valid[j] && st.first[j] && st.ij[j] >= ND)
            ok = ok && wait(bar_de + 8 * (st.ij[j] % ND), (uint32_t)(((st.ij[j] / ND) - 1) & 1));
        if (!ok) break;
        fence_after();
        const uint32_t xb = xring + (uint32_t)((s % kNX) * XSUB);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (!st.valid[j]) continue;
          const uint32_t col = (uint32_t)(DCOLS + 32 * (4 * t + j));
          mma_sp(tmem + (uint32_t)((st.ij[j] % ND) * NPAD), tmem + col + 8,
                 desc_sw128(xb + (uint32_t)((j >> 1) * XBOX + (j & 1) * 64)), tmem + col, IDESC,
                 st.first[j] ? 0u : 1u);
        }
        mma_commit(bar_dn + 8 * (s % kRD));
        s_end = s + 1;
      }
      pub[2 + mine] = s_end;
    }
  } else if (warp >= kEpiWarp0 && warp < kEpiWarp0 + 4) {
    // ======================= epilogue: accumulators -> y ==================
    // Each thread owns one row; its warps never leave the walk early (a wait
    // that runs out just skips ahead), so the named barrier of the split-K
    // hand-off and the per-tile counters always see every epilogue thread.
    const int quad = warp - kEpiWarp0;
    const int r = quad * 32 + lane;
    const int etid = tid - 32 * kEpiWarp0;       // 0..127
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    Walk wk(U, nunits, tile0, uit0);
    int inst = -1;
    bool first_seg = true;
    float acc[NPAD];
#pragma unroll
    for (int i = 0; i < NPAD; ++i) acc[i] = 0.0f;
    for (int s = 0; s < nsub; ++s) {
      const int ui = s / SUBS, ls = s % SUBS;
      if (ls == 0 && ui > 0) wk.next_unit();
      const int seg_u1 = wk.seg_u1(ui);
      const int seg_c1 = min(p.cols, seg_u1 * UNIT_COLS);
      const int scol0 = wk.uit * UNIT_COLS + ls * 128;
      const uint32_t wslot = wring + (uint32_t)((ui % kNW) * kStageW);
      const int g0 = ((wk.uit * UNIT_COLS) >> p.gshift) & ~3;
      Steps st;
      st.walk(scol0, seg_c1, p.group, inst);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (!(st.valid[j] && st.ends[j])) continue;
        const int blk = st.ij[j] % ND;
        __all_sync(0xffffffffu, wait(bar_dn + 8 * (s % kRD), (uint32_t)((s / kRD) & 1)));
        fence_after();
        const int G = (scol0 + 32 * j) >> p.gshift;
        const uint32_t w = lds32(wslot + kSzOff + (uint32_t)(r * 32 + (G - g0) * 4));
        const float sc = __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu)));
        const uint32_t taddr = tmem + lane_off + (uint32_t)(blk * NPAD);
#pragma unroll
        for (int c0 = 0; c0 < NPAD; c0 += 8) {
          uint32_t v0[8];
          ld8(taddr + c0, v0);
          asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[c0 + i] = fmaf(sc, __uint_as_float(v0[i]), acc[c0 + i]);
        }
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_de + 8 * blk);
      }
      if (ls == SUBS - 1) {   // done with the unit's scale words
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_we + 8 * (ui % kNW));
      }
      if (ls == SUBS - 1 && wk.unit_ends_segment(ui)) {
        // ---- the segment is finished: y directly, or through the split-K
        // workspace when the tile is shared with other CTAs
        const int tile = wk.tile;
        const YRow yr(p, tile, r);
        if (wk.seg_u0 == 0 && seg_u1 == U) {
#pragma unroll
          for (int i = 0; i < NPAD; ++i) yr.put(i, p.m, acc[i]);
        } else if (p.parts >= 2) {
          // cluster mode: the partial tile goes to this CTA's own shared
          // memory (the weight ring, free once every epilogue thread has read
          // its last scale word), summed across the cluster after teardown
          asm volatile("bar.sync 1, 128;" ::: "memory");
          float* stage = reinterpret_cast<float*>(sm) + (size_t)r * NPAD;
#pragma unroll
          for (int i = 0; i < NPAD; i += 4)
            *reinterpret_cast<float4*>(stage + i) = make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
        } else {
          const int slot = first_seg ? 0 : 1;
          float* dst = p.scratch + (((size_t)blockIdx.x * 2 + slot) * kRows + r) * NPAD;
#pragma unroll
          for (int i = 0; i < NPAD; i += 4)
            __stcg(reinterpret_cast<float4*>(dst + i),
                   make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]));
          // publish: the named barrier orders every epilogue thread's
          // partial before the arrival, which releases them at GPU scope
          // (and, for the arrival that completes the tile, acquires the
          // other CTAs' partials)
          asm volatile("bar.sync 1, 128;" ::: "memory");
          const long long tu0 = (long long)tile * U, tu1 = tu0 + U - 1;
          const int c0 = (int)(((tu0 + 1) * P - 1) / T), c1 = (int)(((tu1 + 1) * P - 1) / T);
          if (etid == 0) {
            const TcSeg& sg = seg_of(p, tile);
            int* ctr = sg.counters + (tile - sg.tile_begin);
            int old;
            asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;"
                         : "=r"(old)
                         : "l"(ctr)
                         : "memory");
            const bool done = old == c1 - c0;
            if (done) *ctr = 0;   // left at 0 for the next launch
            // the CTA's last segment: the whole CTA sums after its teardown
            // barrier (every role is finished then)
            const bool defer = done && ui + 1 == nunits;
            if (defer) *final_tile = tile;
            *last_flag = done && !defer;
          }
          asm volatile("bar.sync 1, 128;" ::: "memory");
          if (*last_flag) {
            // a tile completed in mid-run: the epilogue threads sum it, one
            // row each, in CTA order
            const int slot0 = split_slot0(c0, tu0, T, P, U);
            float (&sum)[NPAD] = acc;
#pragma unroll
            for (int i = 0; i < NPAD; ++i) sum[i] = 0.0f;
            for (int c = c0; c <= c1; ++c) {
              const float* src =
                  p.scratch + (((size_t)c * 2 + (c == c0 ? slot0 : 0)) * kRows + r) * NPAD;
#pragma unroll
              for (int i = 0; i < NPAD; i += 4) {
                const float4 f = __ldcg(reinterpret_cast<const float4*>(src + i));
                sum[i] += f.x;
                sum[i + 1] += f.y;
                sum[i + 2] += f.z;
                sum[i + 3] += f.w;
              }
            }
#pragma unroll
            for (int i = 0; i < NPAD; ++i) yr.put(i, p.m, sum[i]);
          }
          asm volatile("bar.sync 1, 128;" ::: "memory");   // last_flag is read before it is reused
          first_seg = false;
        }
#pragma unroll
        for (int i = 0; i < NPAD; ++i) acc[i] = 0.0f;
      }
    }
  }

  // ---- teardown.  After an abort: the copies and MMAs this CTA issued are
  // let land (bounded) before its shared and tensor memory are released --
  // only the last load issued into each slot and the last few sub-stages'
  // MMAs can still be in flight.  (The epilogue completed the split-K
  // counters.)
  fence_before();
  __syncthreads();

  // ---- the split-K sum of the tile this CTA completed last, by every
  // thread: float4 groups of the partial tiles in row-major order (coalesced
  // loads), up to 16 partial loads in flight per thread, summed in CTA order
  // like the epilogue's (so y does not depend on which path summed it)
  {
    const int ftile = *final_tile;
    if (ftile >= 0) {
      constexpr int G = NPAD / 4;                  // float4 groups per row
      const long long tu0 = (long long)ftile * U, tu1 = tu0 + U - 1;
      const int c0 = (int)(((tu0 + 1) * P - 1) / T), c1 = (int)(((tu1 + 1) * P - 1) / T);
      const int slot0 = split_slot0(c0, tu0, T, P, U);
      for (int it0 = tid; it0 < kRows * G; it0 += 2 * kThreads) {
        float4 s2[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) s2[k] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        for (int cb = c0; cb <= c1; cb += 8) {
          float4 v[2][8];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int it = it0 + k * kThreads;
            const int r = it / G, g = it % G;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int c = cb + q;
              v[k][q] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
              if (it < kRows * G && c <= c1)
                v[k][q] = __ldcg(reinterpret_cast<const float4*>(
                    p.scratch + (((size_t)c * 2 + (c == c0 ? slot0 : 0)) * kRows + r) * NPAD + 4 * g));
            }
          }
#pragma unroll
          for (int k = 0; k < 2; ++k)
#pragma unroll
            for (int q = 0; q < 8; ++q)
              if (cb + q <= c1) {
                s2[k].x += v[k][q].x;
                s2[k].y += v[k][q].y;
                s2[k].z += v[k][q].z;
                s2[k].w += v[k][q].w;
              }
        }
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int it = it0 + k * kThreads;
          if (it >= kRows * G) continue;
          const int r = it / G, g = it % G;
          const YRow yr(p, ftile, r);
          const float o[4] = {s2[k].x, s2[k].y, s2[k].z, s2[k].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) yr.put(4 * g + q, p.m, o[q]);
        }
      }
    }
  }

  if (tid == 0 && *abort_flag) {
    const unsigned long long lim = p.wait_ns;
    auto settle = [&](uint32_t bar, uint32_t par) {
      const unsigned long long t0 = global_ns();
      while (!mbar_try(bar, par))
        if (global_ns() - t0 > lim) break;
    };
    const int w_issued = pub[0], x_issued = pub[1];
    const int s_mma = pub[2] > pub[3] ? pub[2] : pub[3];
    for (int ui = max(0, w_issued - kNW); ui < w_issued; ++ui)
      settle(bar_wf + 8 * (ui % kNW), (uint32_t)((ui / kNW) & 1));
    for (int x = max(0, x_issued - kNX); x < x_issued; ++x)
      settle(bar_xf + 8 * (x % kNX), (uint32_t)((x / kNX) & 1));
    for (int x = max(0, s_mma - 4); x < s_mma; ++x)
      settle(bar_dn + 8 * (x % kRD), (uint32_t)((x / kRD) & 1));
  }
  __syncthreads();

  // ---- cluster mode: rank q sums rows [q R, (q + 1) R) of the tile, R = 128 /
  // parts, over every rank's staged partial in rank order (the CTA order of
  // the stream-K sum, so y is the same bitwise), reading the other ranks'
  // shared memory directly; a second cluster barrier keeps every CTA's
  // staged tile alive until all ranks have read it.
  if (p.parts >= 2) {
    cluster_sync();
    constexpr int G = NPAD / 4;                   // float4 groups per row
    const int q = (int)(blockIdx.x % p.parts), R = kRows / p.parts;
    const int tile = (int)blockIdx.x / p.parts;
    for (int it = tid; it < R * G; it += kThreads) {
      const int rl = it / G, g = it % G, r = q * R + rl;
      const uint32_t off = base + (uint32_t)((r * G + g) * 16);
      float4 sum = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      for (int k0 = 0; k0 < p.parts; k0 += 4) {
        float4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          v[k] = k0 + k < p.parts ? ld_cluster_f4(mapa_rank(off, (uint32_t)(k0 + k)))
                                  : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (k0 + k < p.parts) {
            sum.x += v[k].x;
            sum.y += v[k].y;
            sum.z += v[k].z;
            sum.w += v[k].w;
          }
      }
      const YRow yr(p, tile, r);
      const float o[4] = {sum.x, sum.y, sum.z, sum.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) yr.put(4 * g + k, p.m, o[k]);
    }
    cluster_sync();
  }
  if (warp == kMmaWarp) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols)
                 : "memory");
  }
}

}  // namespace
}  // namespace sgemv

// ---- host side --------------------------------------------------------------
namespace sgemv {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

// A 2-D map over a row-major array of `rows` rows of `inner` elements.
bool encode_2d(CUtensorMap* map, CUtensorMapDataType dt, int esize, const void* ptr,
               uint64_t inner, uint64_t rows, uint32_t box_inner, uint32_t box_rows,
               CUtensorMapSwizzle sw, CUtensorMapL2promotion l2) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || !ptr || inner == 0 || rows == 0) return false;
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {inner * (uint64_t)esize};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, sw, l2, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int g_tc_sms[64] = {0};

int tc_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!g_tc_sms[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_tc_sms[dev] = n;
  }
  return g_tc_sms[dev];
}

int npad_of(int m) { return ((m + 15) / 16) * 16; }

size_t tc_smem(int npad) {
  // 1024 alignment slack + weight ring + x ring + barriers and flags (at
  // most 8 * (2 kNW + kNX + NA + kRD + ND) + 28 bytes); at
  // least 120 KB, so that one CTA (and one tensor-memory allocation) per SM
  const size_t need = 1024 + (size_t)kNW * kStageW + (size_t)kNX * 2 * npad * 128 + 1024;
  return need < 120 * 1024 ? 120 * 1024 : need;
}

// One launch over `count` matrices that share x, cols, N, the group size and
// m; the split-K partials go to maps[0]'s workspace, each matrix's tile
// arrivals to its own counters.
template <int N, int NPAD>
cudaError_t launch_tc_n(const Layout* Ls, const RunArgs* as, const TcMaps* const* maps, int count,
                        cudaStream_t s, int max_ctas) {
  constexpr int UNIT_COLS = N == 2 ? 256 : 512;
  const int sms = tc_sms();
  if (sms <= 0) return cudaErrorNotSupported;
  const Layout& L = Ls[0];
  const RunArgs& a = as[0];
  TcParams p;
  memset(&p, 0, sizeof p);
  int ntiles = 0;
  for (int i = 0; i < count; ++i) {
    TcSeg& sg = p.seg[i];
    sg.tm_vals = maps[i]->vals;
    sg.tm_idx = maps[i]->idx;
    sg.tm_sz = maps[i]->sz;
    sg.y = as[i].y;
    sg.counters = maps[i]->counters;
    sg.rows = Ls[i].rows;
    sg.tile_begin = ntiles;
    ntiles += (Ls[i].rows + kRows - 1) / kRows;
  }
  for (int i = count; i < kTcMaxSeg; ++i) p.seg[i].tile_begin = ntiles;
  p.nseg = count;
  if (!encode_2d(&p.tm_x, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.x, (uint64_t)L.cols,
                 (uint64_t)a.m, 64, NPAD, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_128B))
    return cudaErrorInvalidValue;
  p.scratch = maps[0]->scratch;
  p.err = a.err;
  p.cols = L.cols;
  p.m = a.m;
  p.group = L.group;
  p.gshift = L.group == 64 ? 6 : (L.group == 128 ? 7 : 8);
  p.ntiles = ntiles;
  p.units_per_tile = (L.cols + UNIT_COLS - 1) / UNIT_COLS;
  p.total_units = (long long)p.ntiles * p.units_per_tile;
  const int cap = sms < max_ctas ? sms : max_ctas;
  // cluster mode when every tile fits 2..8 CTAs (a power of two, at least
  // one unit each) within the SMs: no workspace, no counters, no CTA waiting
  // on a global arrival
  p.parts = 0;
  if (kClusterMode && p.ntiles <= cap) {
    int parts = cap / p.ntiles;
    parts = parts > 8 ? 8 : parts;
    parts = parts > p.units_per_tile ? p.units_per_tile : parts;
    while (parts & (parts - 1)) parts &= parts - 1;
    if (parts >= 2) p.parts = parts;
  }
  p.grid = (int)(p.total_units < cap ? p.total_units : cap);
  // A grid whose equal unit runs fall on tile boundaries -- k units per CTA
  // with k dividing the tile's units (each tile shared by exactly U / k CTAs,
  // no CTA straddling two) or a multiple of them (no split at all) -- when
  // one exists with at least kAlignPct% of the CTAs: fewer partial tiles and
  // no split-K publication in mid-run, for some idle SMs.  (Measured on the
  // config-4 layer set: the 11008-row layers run faster on 86 CTAs of one
  // whole tile each than on 152 sharing tiles, by 7% of the step at M = 64.)
  if (p.parts >= 2) p.grid = p.ntiles * p.parts;
  if (p.parts < 2 && kAlignPct > 0 && p.total_units > p.grid && p.total_units % p.grid != 0) {
    for (int g = p.grid - 1; 100 * g >= kAlignPct * p.grid; --g) {
      if (p.total_units % g) continue;
      const long long k = p.total_units / g;
      if (p.units_per_tile % k == 0 || k % p.units_per_tile == 0) {
        p.grid = g;
        break;
      }
    }
  }
  p.withhold = a.withhold;
  p.wait_ns = a.withhold ? kInjectWaitNs : kWaitLimitNs;
  const size_t smem = tc_smem(NPAD);
  static bool attr_set[64] = {false};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(k_tc<N, NPAD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         227 * 1024);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = p.parts >= 2 ? p.parts : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.parts >= 2 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k_tc<N, NPAD>, p);
}

}  // namespace

size_t tc_scratch_bytes(int max_m) {
  if (max_m < 2) return 0;
  const int sms = tc_sms();
  return (size_t)(sms > 0 ? sms : 0) * 2 * kRows * npad_of(max_m) * sizeof(float);
}

int tc_tiles(const Layout& L) { return (L.rows + kRows - 1) / kRows; }

bool tc_encode_weights(const Layout& L, const uint4* vals, const uint2* idx, const uint32_t* sz,
                       TcMaps* maps) {
  if (L.rows == 0 || L.cols == 0) return false;
  return encode_2d(&maps->vals, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, vals, (uint64_t)L.cstride * 16,
                   (uint64_t)L.rows, 64, kRows, CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B) &&
         encode_2d(&maps->idx, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, idx, (uint64_t)L.cstride * 8,
                   (uint64_t)L.rows, 32, kRows, CU_TENSOR_MAP_SWIZZLE_32B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B) &&
         encode_2d(&maps->sz, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, sz, (uint64_t)L.gstride,
                   (uint64_t)L.rows, kSzWords, kRows, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_128B);
}

cudaError_t launch_tc(const Layout& L, const RunArgs& a, const TcMaps& maps, cudaStream_t s) {
  return launch_tc(L, a, maps, s, 1 << 30);
}

cudaError_t launch_tc(const Layout& L, const RunArgs& a, const TcMaps& maps, cudaStream_t s,
                      int max_ctas) {
  const TcMaps* m[1] = {&maps};
  return launch_tc_group(&L, &a, m, 1, s, max_ctas);
}

int tc_max_group() { return kTcMaxSeg; }

cudaError_t launch_tc_group(const Layout* Ls, const RunArgs* as, const TcMaps* const* maps,
                            int count, cudaStream_t s, int max_ctas) {
  if (max_ctas < 1) return cudaErrorInvalidValue;
  if (count < 1 || count > kTcMaxSeg) return cudaErrorNotSupported;
  const Layout& L = Ls[0];
  const RunArgs& a = as[0];
  if (a.m < 2 || a.m > 64 || !maps[0]->scratch) return cudaErrorNotSupported;
  for (int i = 0; i < count; ++i)
    if (Ls[i].rows == 0 || Ls[i].cols != L.cols || Ls[i].cols == 0 ||
        Ls[i].n_keep != L.n_keep || Ls[i].group != L.group || as[i].m != a.m ||
        as[i].x != a.x || !maps[i]->ready || !maps[i]->counters)
      return cudaErrorNotSupported;
  if (((uintptr_t)a.x & 15u) != 0) return cudaErrorNotSupported;
  const int np = npad_of(a.m);
  if (L.n_keep == 2) {
    switch (np) {
      case 16: return launch_tc_n<2, 16>(Ls, as, maps, count, s, max_ctas);
      case 32: return launch_tc_n<2, 32>(Ls, as, maps, count, s, max_ctas);
      case 48: return launch_tc_n<2, 48>(Ls, as, maps, count, s, max_ctas);
      default: return launch_tc_n<2, 64>(Ls, as, maps, count, s, max_ctas);
    }
  }
  switch (np) {
    case 16: return launch_tc_n<1, 16>(Ls, as, maps, count, s, max_ctas);
    case 32: return launch_tc_n<1, 32>(Ls, as, maps, count, s, max_ctas);
    case 48: return launch_tc_n<1, 48>(Ls, as, maps, count, s, max_ctas);
    default: return launch_tc_n<1, 64>(Ls, as, maps, count, s, max_ctas);
  }
}

}  // namespace sgemv
