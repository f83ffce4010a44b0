// Causal softmax attention forward on sm_103a, with optional on-chip RoPE of the Q and K tiles.
//
// What it computes: for every batch b, query head h (KV head h / (Hq/Hkv)) and query row i,
//   o_i = sum_{j <= i} softmax_j(q'_i . k'_j / sqrt(d)) v_j   and   lse_i = ln sum_{j<=i} exp(...),
// (with Nk > N keys the queries are the last N tokens and the sums run over j <= Nk - N + i),
// where q', k' are RoPE-rotated (fused mode) or were rotated beforehand (pre-rotate mode: the
// kernel then runs with ROTATE = false on already-rotated inputs).  RoPE is a pre-multiplication
// transform and the causal mask and softmax are building blocks of one fused kernel ("AttnFuse Makes
// RoPE a First-Class Attention Compilation Operation", 2026-09-13 AI papers report, paragraphs 1-2).
// The online softmax keeps a running row max m_i and denominator l_i ("Fast and Exact
// Relative-Position Attention via Structure-Aware Kernels", prerequisites: FlashAttention and
// online softmax), in fp32 and with base-2 exponentials (same page, technical novelty (4)).
//
// Structure: persistent, one CTA (512 threads) per SM walking a list of work units; a unit is two
// 128-row query tiles q0, q1 that share every K and V tile: two heads of one KV group on the same
// rows when the group size is even, else two consecutive row blocks of one head.
//   warp 0        TMA producer: per unit Q, and K and V tiles (128 keys) through 2-stage rings.
//   warp 1        tcgen05.mma issuer; owns the tensor-memory allocation (512 columns:
//                 S0 | S1 | O0 | O1, P_i written over the first half of S_i).
//   warps 4-7     softmax for q0 (thread = query row = TMEM lane), epilogue for q0.
//   warps 8-11    softmax for q1, epilogue for q1.
//   warps 12-15   fused mode: rotate the Q tiles and every K tile in shared memory before their
//                 QK^T MMAs.
// MMA order per key tile i: S0_i, PV1_{i-1}, S1_i, PV0_i, so that each softmax warpgroup works on
// one tile while the tensor cores run the other's products; the pending PV1 of a unit's last tile
// is issued after the next unit's first S0, and the next unit's Q is loaded as soon as the last
// QK^T of the current unit is done with the Q buffer.  Fully masked key tiles are never
// loaded (tile i runs for query tile qt only while i <= qt); the diagonal tile is masked per
// element.  The softmax takes a row's max from its first key tile only and computes every later
// tile's P against that running max, without a max pass; only when a row of P sums past 2^15 (a
// score outgrew the max by ~15 in log2 units) is that tile redone with its own max and O and l
// rescaled.  The result stays exact: the max used is applied consistently to P, l and lse.
//
// Every barrier wait gives up after AttnParams::timeout_ns: the CTA then records bit 0 in the
// device status word, stops its loops, lets its copies and MMAs land, frees tensor memory and
// returns.  Later CTAs see the status word and return at once.
#include <cuda_runtime.h>
#include <math.h>

#include <type_traits>

#include "attnfuse_internal.h"
#include "ptx.cuh"
#include "rope.cuh"

namespace attnfuse {

__device__ unsigned int g_device_status = 0;

namespace {

constexpr int BM = 128;  // query rows per tile (= TMEM lanes)
constexpr int BN = 128;  // keys per tile
constexpr int kThreads = 512;
constexpr int KST = 2;   // K ring depth
constexpr int VST = 2;   // V ring depth
constexpr uint32_t kBoxBytes = 128 * 128;  // 128 rows x 64 16-bit columns, 128-byte swizzled
constexpr uint32_t kTmemCols = 512;
constexpr float kLn2 = 0.6931471805599453f;
// A tile's P = 2^(s - m) is computed with the running max m of the earlier tiles; only when some row
// of P sums past this bound (some score exceeded m by more than ~15 in log2 units, so P could leave
// the range of the 16-bit operand type) is the tile redone with its own max.
constexpr float kSumCap = 32768.0f;

// Register split after setmaxnreg (control warps / softmax warps / rotation warps).  The total,
// 128 x (ctrl + rotate) + 256 x softmax, must not exceed the 512 x 128 registers the CTA is launched
// with, or the softmax warps' setmaxnreg.inc would wait forever.
template <int D, bool ROTATE>
struct Regs {
  // Without rotation the rotation warps are idle and the softmax warps take their registers.
  static constexpr uint32_t kCtrl = ROTATE ? 88 : 80;
  static constexpr uint32_t kSoftmax = ROTATE ? 168 : 176;
  static constexpr uint32_t kRotate = ROTATE ? 88 : 80;
  static_assert(128 * (kCtrl + kRotate) + 256 * kSoftmax <= kThreads * 128, "register split");
};

// Row max of 128 scores held as fp32 bit patterns: three-input max tree, eight independent chains.
__device__ __forceinline__ float row_max128(const uint32_t (&sv)[4][32]) {
  float acc[8];
#pragma unroll
  for (int k = 0; k < 8; ++k)
    acc[k] = ptx::fmax3(__uint_as_float(sv[0][k]), __uint_as_float(sv[0][k + 8]), __uint_as_float(sv[0][k + 16]));
#pragma unroll
  for (int base = 24; base < 120; base += 16)
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i0 = base + k, i1 = base + 8 + k;
      acc[k] = ptx::fmax3(acc[k], __uint_as_float(sv[i0 / 32][i0 % 32]), __uint_as_float(sv[i1 / 32][i1 % 32]));
    }
#pragma unroll
  for (int k = 0; k < 8; ++k) acc[k] = fmaxf(acc[k], __uint_as_float(sv[3][24 + k]));
  return ptx::fmax3(ptx::fmax3(acc[0], acc[1], acc[2]), ptx::fmax3(acc[3], acc[4], acc[5]), fmaxf(acc[6], acc[7]));
}

// P = 2^(s * sl2 - m) for one row of 128 scores on fp32 pairs, packed to the operand type into
// pk (64 words); returns the row sum (four independent partials).
template <bool BF16>
__device__ __forceinline__ float softmax_p(const uint32_t (&sv)[4][32], float sl2, float m, uint32_t (&pk)[64]) {
  const uint64_t SL2 = ptx::f2_pack(sl2, sl2), NM = ptx::f2_pack(-m, -m);
  uint64_t part[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) part[k] = ptx::f2_pack(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < 4; ++c) {  // S columns [32 c, 32 c + 32) -> P words [16 c, 16 c + 16)
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const uint64_t x2 =
          ptx::f2_fma(ptx::f2_pack(__uint_as_float(sv[c][2 * e]), __uint_as_float(sv[c][2 * e + 1])), SL2, NM);
      float x0, x1;
      ptx::f2_unpack(x2, x0, x1);
      const float p0 = ptx::ex2_approx(x0), p1 = ptx::ex2_approx(x1);
      part[e & 3] = ptx::f2_add(part[e & 3], ptx::f2_pack(p0, p1));
      pk[16 * c + e] = Pack<BF16>::pack(p0, p1);
    }
  }
  float a, b;
  ptx::f2_unpack(ptx::f2_add(ptx::f2_add(part[0], part[1]), ptx::f2_add(part[2], part[3])), a, b);
  return a + b;
}

// Rare path of the softmax, taken by a whole warp when some row's P summed past kSumCap (its scores
// outgrew the running max): rows with `need` take the tile's own max, rescale l and O, and P is
// recomputed from S (still intact in tensor memory) and stored.  Returns the row sum and the updated
// max and denominator.  Kept out of line so that the common path's register allocation does not
// carry it.
struct RowState {
  float sum, m, l;
};
template <int D, bool BF16>
__device__ __noinline__ RowState softmax_redo(uint32_t tS, uint32_t tO, int lim, bool diag, bool need, float sl2,
                                              float m_run, float l_run) {
  float mx = -INFINITY;
  for (int c = 0; c < 8; ++c) {
    uint32_t t[16];
    ptx::tmem_ld16(tS + 16 * c, t);
    ptx::tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 16; ++e)
      if (!(diag && 16 * c + e > lim)) mx = fmaxf(mx, __uint_as_float(t[e]));
  }
  float alpha = 1.f;
  if (need) {
    const float m_new = fmaxf(m_run, mx * sl2);
    alpha = ptx::ex2_approx(m_run - m_new);
    l_run *= alpha;
    m_run = m_new;
  }
  // The previous O += P V finished before s_full; this tile's waits for p_full.
  for (int c = 0; c < D / 16; ++c) {
    uint32_t o[16];
    ptx::tmem_ld16(tO + 16 * c, o);
    ptx::tmem_wait_ld();
#pragma unroll
    for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
    ptx::tmem_st16(tO + 16 * c, o);
  }
  const float nm = -m_run;
  float sum = 0.f;
  for (int c = 0; c < 4; ++c) {  // S columns [32 c, 32 c + 32) -> P words [16 c, 16 c + 16) (columns
    uint32_t pk[16];              // already read: the loads run ahead of the stores)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t t[16];
      ptx::tmem_ld16(tS + 32 * c + 16 * h, t);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int col = 32 * c + 16 * h + 2 * e;
        const float x0 = (diag && col > lim) ? -INFINITY : fmaf(__uint_as_float(t[2 * e]), sl2, nm);
        const float x1 = (diag && col + 1 > lim) ? -INFINITY : fmaf(__uint_as_float(t[2 * e + 1]), sl2, nm);
        const float p0 = ptx::ex2_approx(x0), p1 = ptx::ex2_approx(x1);
        sum += p0 + p1;
        pk[8 * h + e] = Pack<BF16>::pack(p0, p1);
      }
    }
    ptx::tmem_st16(tS + 16 * c, pk);
  }
  return RowState{sum, m_run, l_run};
}

template <int D>
struct Cfg {
  static constexpr int NBOX = D / 64;
  static constexpr uint32_t TILE = NBOX * kBoxBytes;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + 2 * TILE;
  static constexpr uint32_t OFF_V = OFF_K + KST * TILE;
  static constexpr uint32_t OFF_CTL = OFF_V + VST * TILE;
  static constexpr uint32_t OFF_FREQ = OFF_CTL + 256;     // F_k words: lo[64] then hi[64]
  static constexpr uint32_t SMEM = OFF_FREQ + 512 + 1024;  // + alignment slack
  static constexpr uint32_t COL_O = 2 * BN;               // O0 at 256, O1 at 256 + D
  static_assert(COL_O + 2 * D <= kTmemCols, "TMEM budget");
};

struct __align__(8) Ctrl {
  uint64_t q_full, q_empty;
  uint64_t q_ready[2];  // query tile i rotated (by softmax warpgroup i)
  uint64_t k_full[KST], k_ready[KST], k_empty[KST];
  uint64_t v_full[VST], v_empty[VST];
  uint64_t s_full[2], p_full[2], o_full[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
  int skip;
  int q_off;  // AttnParams::q_off
};
static_assert(sizeof(Ctrl) <= 256, "control block");

__device__ __forceinline__ uint32_t bar_addr(const uint64_t& b) { return ptx::smem_u32(&b); }

__device__ __forceinline__ void signal_abort(Ctrl& ctl) {
  *reinterpret_cast<volatile int*>(&ctl.abort_flag) = 1;
  atomicOr(&g_device_status, 1u);
}

// Bounded wait; false if it ran out (and raised the abort) or another thread aborted.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, Ctrl& ctl, unsigned long long timeout_ns) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*reinterpret_cast<volatile int*>(&ctl.abort_flag)) return false;
      if (ptx::globaltimer_ns() - t0 > timeout_ns) {
        signal_abort(ctl);
        return false;
      }
    }
  }
}

// Bounded wait that ignores the abort flag: used only to let in-flight copies and MMAs land.
__device__ __forceinline__ bool drain_bar(uint32_t bar, uint32_t parity, unsigned long long timeout_ns) {
  const uint64_t t0 = ptx::globaltimer_ns();
  for (;;) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    if (ptx::globaltimer_ns() - t0 > timeout_ns) return false;
  }
}

// Whole-warp wait with a warp-uniform outcome: every lane polls (so every lane gets acquire
// ordering from its own successful try_wait) and a vote makes the result the same for the warp.
// (Polling by lane 0 alone with the outcome broadcast measured slower.)
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, Ctrl& ctl,
                                              unsigned long long timeout_ns) {
  bool ok = wait_bar(bar, parity, ctl, timeout_ns);
  return __all_sync(0xFFFFFFFFu, ok);
}

// The MMA issuer's instructions in its two forms.  Issue<true>: the whole warp runs the issuing
// role (control flow and operands warp-uniform, barrier waits by the warp, one elected lane
// issues); Issue<false>: one lane runs it alone.  Measured on GB300 at the Llama-3-8B shape, the
// warp form issues a 128x128x16 MMA in ~35 cycles against ~58 and makes the plain attention kernel
// 4% faster, but the rotating kernel 1.6% slower, so each kernel takes the faster form.
template <bool WARP>
struct Issue {
  static __device__ __forceinline__ void ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    if constexpr (WARP) ptx::mma_ss_w(d, a, b, idesc, acc); else ptx::mma_ss(d, a, b, idesc, acc);
  }
  static __device__ __forceinline__ void ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    if constexpr (WARP) ptx::mma_ts_w(d, a, b, idesc, acc); else ptx::mma_ts(d, a, b, idesc, acc);
  }
  static __device__ __forceinline__ void commit(uint32_t bar) {
    if constexpr (WARP) ptx::mma_commit_w(bar); else ptx::mma_commit(bar);
  }
  static __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, Ctrl& ctl, unsigned long long tmo) {
    if constexpr (WARP) return wait_bar_warp(bar, parity, ctl, tmo); else return wait_bar(bar, parity, ctl, tmo);
  }
};

// Byte offsets, inside a 128-row tile of 128-byte swizzled boxes, of the two 16-byte chunks that
// hold the rotation pairs (k, k + d/2) for k in [8 ck, 8 ck + 8) of row r.  TMA's 128-byte
// swizzle stores logical chunk c of row r at physical chunk c ^ (r & 7).
template <int D>
__device__ __forceinline__ void pair_offsets(int r, int ck, uint32_t& xo, uint32_t& yo) {
  if constexpr (D == 128) {
    xo = (uint32_t)r * 128u + (uint32_t)((ck ^ (r & 7)) * 16);
    yo = xo + kBoxBytes;  // columns 64..127 live in the second box at the same offset
  } else {
    xo = (uint32_t)r * 128u + (uint32_t)((ck ^ (r & 7)) * 16);
    yo = (uint32_t)r * 128u + (uint32_t)(((ck + 4) ^ (r & 7)) * 16);
  }
}

// Thread -> (chunk ck, first row r0) for rotating a 128-row tile with 128 threads: a thread keeps one
// chunk (8 frequencies) and walks rows r0, r0 + RS, ... (RS = 16 for d = 128, 32 for d = 64).  Eight
// consecutive lanes cover eight distinct 16-byte chunks of one 128-byte row (d = 128) or two rows
// whose swizzle differs by 4 (d = 64), so every 16-byte shared access is free of bank conflicts.
template <int D>
__device__ __forceinline__ void rot_mapping(int rt, int& ck, int& r0) {
  const int w = rt >> 5, lane = rt & 31;
  if constexpr (D == 128) {
    ck = lane & 7;
    r0 = w * 4 + (lane >> 3);
  } else {
    ck = lane & 3;
    const int q = lane >> 2;
    r0 = w * 8 + (((q & 1) << 2) | (q >> 1));
  }
}

template <int D>
struct RotGeom {
  static constexpr int PASSES = D == 128 ? 8 : 4;
  static constexpr int RS = 128 / PASSES;
};

// Rotate, in place, the thread's rows of one 128-row tile held in shared memory at `tile`.  On entry
// cs holds the cos/sin of the thread's first row r0; it is advanced by `step` (the exact rotation of
// RS rows) after every pass, so on return it holds the values of row r0 + 128 -- the thread's first
// row of the next tile.
template <int D, bool BF16>
__device__ __forceinline__ void rotate_tile(uint32_t tile, int r0, int ck, RopeCS8& cs, const RopeCS8& step) {
  constexpr int PASSES = RotGeom<D>::PASSES, RS = RotGeom<D>::RS;
#pragma unroll
  for (int pass = 0; pass < PASSES; pass += 2) {
    uint32_t xo0, yo0, xo1, yo1;
    pair_offsets<D>(r0 + pass * RS, ck, xo0, yo0);
    pair_offsets<D>(r0 + (pass + 1) * RS, ck, xo1, yo1);
    uint4 x0 = ptx::lds128(tile + xo0), y0 = ptx::lds128(tile + yo0);
    uint4 x1 = ptx::lds128(tile + xo1), y1 = ptx::lds128(tile + yo1);
    rope_rotate_chunk_cs8<BF16>(x0, y0, cs);
    rope_cs8_advance(cs, step);
    rope_rotate_chunk_cs8<BF16>(x1, y1, cs);
    rope_cs8_advance(cs, step);
    ptx::sts128(tile + xo0, x0);
    ptx::sts128(tile + yo0, y0);
    ptx::sts128(tile + xo1, x1);
    ptx::sts128(tile + yo1, y1);
  }
}

// Byte offset, inside a 128-row tile of 128-byte swizzled boxes, of 16-byte chunk c (elements
// [8c, 8c + 8)) of row r: box c / 8, logical chunk c % 8 stored at physical chunk (c % 8) ^ (r & 7).
__device__ __forceinline__ uint32_t chunk_offset(int r, int c) {
  return (uint32_t)(c >> 3) * kBoxBytes + (uint32_t)r * 128u + (uint32_t)((((c & 7) ^ (r & 7))) * 16);
}

// rotate_tile for the RoPE variants: the thread's chunk pair ck works only if ck < R (= rotary_dim
// / 16); its chunks are ck and ck + R (pairs (k, k + rotary_dim/2)) or the adjacent 2 ck, 2 ck + 1
// (pairs (2k, 2k + 1)), with frequencies 8 ck .. 8 ck + 7 either way.  With pos == nullptr the
// rows take the carried cos/sin walk of rotate_tile; otherwise row r of the tile sits at position
// pos[r] (rows r >= nvalid, past the end of the sequence, at 0) and its cos/sin are computed exactly.
template <int D, bool BF16>
__device__ __forceinline__ void rotate_tile_variant(uint32_t tile, int r0, int ck, RopeCS8& cs, const RopeCS8& step,
                                                    int R, bool interleaved, const int32_t* pos, int nvalid,
                                                    const uint32_t* sfreq) {
  constexpr int PASSES = RotGeom<D>::PASSES, RS = RotGeom<D>::RS;
  if (ck >= R) return;
  const int ca = interleaved ? 2 * ck : ck, cb = interleaved ? 2 * ck + 1 : ck + R;
  auto rotate_row = [&](int row, const RopeCS8& c8) {
    const uint32_t xo = chunk_offset(row, ca), yo = chunk_offset(row, cb);
    uint4 x = ptx::lds128(tile + xo), y = ptx::lds128(tile + yo);
    if (interleaved) {
      rope_rotate_chunk_il_cs8<BF16>(x, c8, 0);
      rope_rotate_chunk_il_cs8<BF16>(y, c8, 1);
    } else {
      rope_rotate_chunk_cs8<BF16>(x, y, c8);
    }
    ptx::sts128(tile + xo, x);
    ptx::sts128(tile + yo, y);
  };
  if (pos != nullptr) {
    int32_t m[PASSES];
#pragma unroll
    for (int pass = 0; pass < PASSES; ++pass) {
      const int row = r0 + pass * RS;
      m[pass] = row < nvalid ? __ldg(pos + row) : 0;
    }
#pragma unroll 1
    for (int pass = 0; pass < PASSES; ++pass) {
      RopeCS8 c8;
      rope_cs8_exact_signed(m[pass], sfreq, sfreq + 64, ck * 8, c8);
      rotate_row(r0 + pass * RS, c8);
    }
    return;
  }
#pragma unroll
  for (int pass = 0; pass < PASSES; ++pass) {
    rotate_row(r0 + pass * RS, cs);
    rope_cs8_advance(cs, step);
  }
}

// ---- persistent schedule -------------------------------------------------------------------
// Work unit = (b, head pair, 128-row block t) or (b, h, 256-row block t), numbered longest-first
// (t descending).  CTA c of G
// processes units c, 2G-1-c, 2G+c, 4G-1-c, ... (a snake over the longest-first order), which evens
// out the causal work across CTAs without a shared counter.  Every role walks the same sequence.
struct Unit {
  int b, hk, n0, n1, n_kt;
  int h0, h1, r0, r1;  // query tile i: head h_i, first row r_i
  bool active1;
  __device__ __forceinline__ int head(int i) const { return i == 0 ? h0 : h1; }
  __device__ __forceinline__ int row(int i) const { return i == 0 ? r0 : r1; }
};

__device__ __forceinline__ int unit_of_round(int round, int c, int G) {
  return round * G + ((round & 1) ? (G - 1 - c) : c);
}

// The k-th unit of this CTA (the sequence FOR_EACH_UNIT walks), or -1 after its last.
__device__ __forceinline__ int unit_at(int k, const AttnParams& p) {
  if (k * (int)gridDim.x >= p.total_units) return -1;
  const int u = unit_of_round(k, blockIdx.x, gridDim.x);
  return u < p.total_units ? u : -1;
}

// Key tiles a query tile starting at row r needs: its last row r' = min(r + 127, N - 1) sees keys
// up to q_off + r'.  With q_off = 0 (GENERAL = false) that is t + 1 for the tile starting at 128 t.
template <bool GENERAL>
__device__ __forceinline__ int key_tiles(int r, const AttnParams& p) {
  if constexpr (GENERAL) return (p.q_off + min(r + BM - 1, p.N - 1)) / BN + 1;
  return r / BM + 1;
}

template <bool GENERAL>
__device__ __forceinline__ Unit decode_unit(int u, const AttnParams& p) {
  Unit x;
  if (p.head_pairs) {
    // Two query heads of one KV group on the same 128 rows: q0 = head 2 j, q1 = head 2 j + 1, both
    // over the same key tiles.
    const int pairs = p.B * (p.Hq / 2);
    const int t = p.n_qblocks - 1 - u / pairs;
    const int bj = u - (u / pairs) * pairs;
    x.b = bj / (p.Hq / 2);
    x.h0 = 2 * (bj - x.b * (p.Hq / 2));
    x.h1 = x.h0 + 1;
    x.hk = x.h0 / (p.Hq / p.Hkv);
    x.r0 = x.r1 = t * BM;
    x.active1 = true;
    x.n0 = x.n1 = x.n_kt = key_tiles<GENERAL>(x.r0, p);
    return x;
  }
  // Two consecutive 128-row tiles of one head: q0 rows 256 t.., q1 rows 256 t + 128..
  const int bh_count = p.B * p.Hq;
  const int t = p.n_qblocks - 1 - u / bh_count;
  const int bh = u - (u / bh_count) * bh_count;
  x.b = bh / p.Hq;
  x.h0 = x.h1 = bh - x.b * p.Hq;
  x.hk = x.h0 / (p.Hq / p.Hkv);
  x.r0 = t * 2 * BM;
  x.r1 = x.r0 + BM;
  x.active1 = x.r1 < p.N;
  x.n0 = key_tiles<GENERAL>(x.r0, p);                     // key tiles for q0
  x.n1 = x.active1 ? key_tiles<GENERAL>(x.r1, p) : 0;  // key tiles for q1
  x.n_kt = x.active1 ? x.n1 : x.n0;
  return x;
}

#define FOR_EACH_UNIT(U)                                                         \
  for (int rnd_ = 0; rnd_ * (int)gridDim.x < p.total_units; ++rnd_)             \
    if (const int u_ = unit_of_round(rnd_, blockIdx.x, gridDim.x); u_ >= p.total_units) \
      break;                                                                     \
    else if (const Unit U = decode_unit<VARIANT>(u_, p); true)

template <int D, bool ROTATE, bool BF16, bool VARIANT, bool ROT_K>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ AttnParams p) {
  using C = Cfg<D>;
  using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
  constexpr uint32_t AB = BF16 ? 1u : 0u;
  constexpr uint32_t IDESC_S = ptx::idesc_f16(AB, BM, BN, 0, 0);   // S = Q K^T: A, B K-major
  constexpr uint32_t IDESC_PV = ptx::idesc_f16(AB, BM, D, 0, 1);   // O += P V: B (V) MN-major

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* sgen = smem_raw + (sbase - raw);
  Ctrl& ctl = *reinterpret_cast<Ctrl*>(sgen + C::OFF_CTL);
  const uint32_t sQ = sbase + C::OFF_Q, sK = sbase + C::OFF_K, sV = sbase + C::OFF_V;

  const int warp = __shfl_sync(0xFFFFFFFFu, (int)(threadIdx.x / 32), 0);  // warp-uniform for the compiler
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar_addr(ctl.q_full), 1);
    for (int i = 0; i < 2; ++i) ptx::mbar_init(bar_addr(ctl.q_ready[i]), 128);
    ptx::mbar_init(bar_addr(ctl.q_empty), 1);
    for (int s = 0; s < KST; ++s) {
      ptx::mbar_init(bar_addr(ctl.k_full[s]), 1);
      ptx::mbar_init(bar_addr(ctl.k_ready[s]), 128);
      ptx::mbar_init(bar_addr(ctl.k_empty[s]), 1);
    }
    for (int s = 0; s < VST; ++s) {
      ptx::mbar_init(bar_addr(ctl.v_full[s]), 1);
      ptx::mbar_init(bar_addr(ctl.v_empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bar_addr(ctl.s_full[i]), 1);
      ptx::mbar_init(bar_addr(ctl.p_full[i]), 128);
      ptx::mbar_init(bar_addr(ctl.o_full[i]), 1);
    }
    ptx::mbar_init(bar_addr(ctl.mma_done), 1);
    ctl.abort_flag = 0;
    ctl.q_off = p.q_off;
    ctl.skip = (*reinterpret_cast<volatile unsigned int*>(&g_device_status)) != 0u;
    ptx::fence_barrier_init();
    ptx::fence_proxy_async_smem();
  }
  uint32_t* sfreq = reinterpret_cast<uint32_t*>(sgen + C::OFF_FREQ);
  if (ROTATE && threadIdx.x >= 128 && threadIdx.x < 256) {
    const int k = threadIdx.x - 128;
    sfreq[k] = k < 64 ? p.freqs.lo[k] : p.freqs.hi[k - 64];
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_u32(&ctl.tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  const bool skip = __shfl_sync(0xFFFFFFFFu, ctl.skip, 0) != 0;
  const unsigned long long tmo = p.timeout_ns;
  __syncwarp();  // setmaxnreg and tcgen05 warp-collectives need converged warps

  if (warp < 4) {
    ptx::setmaxnreg_dec<Regs<D, ROTATE>::kCtrl>();
    if (!skip && warp == 0 && lane == 0) {
      // ================================ TMA producer ==========================================
      // Per unit: K_0/V_0 first (their ring stages free up early), then Q once the previous
      // unit's QK^T products are done with the Q buffer, then the remaining K/V tiles.
      ptx::tma_prefetch_desc(&tmQ);
      ptx::tma_prefetch_desc(&tmK);
      ptx::tma_prefetch_desc(&tmV);
      // After a pre-rotation pass (pre-rotate and split modes) this launch may start early; nothing
      // that pass writes is read before this point.
      if constexpr (!(ROTATE && ROT_K)) ptx::grid_dep_wait();
      int gk = 0, gv = 0, uc = 0;
      bool ok = true;
      FOR_EACH_UNIT(U) {
        auto load_kv = [&](int i) -> bool {
          const int ks = gk % KST, kph = (gk / KST) & 1;
          if (!wait_bar(bar_addr(ctl.k_empty[ks]), kph ^ 1, ctl, tmo)) return false;
          ptx::mbar_arrive_expect_tx(bar_addr(ctl.k_full[ks]), C::TILE);
          for (int bx = 0; bx < C::NBOX; ++bx)
            ptx::tma_load_4d(sK + ks * C::TILE + bx * kBoxBytes, &tmK, bar_addr(ctl.k_full[ks]), bx * 64, U.hk,
                             i * BN, U.b);
          ++gk;
          const int vs = gv % VST, vph = (gv / VST) & 1;
          if (!wait_bar(bar_addr(ctl.v_empty[vs]), vph ^ 1, ctl, tmo)) return false;
          ptx::mbar_arrive_expect_tx(bar_addr(ctl.v_full[vs]), C::TILE);
          for (int bx = 0; bx < C::NBOX; ++bx)
            ptx::tma_load_4d(sV + vs * C::TILE + bx * kBoxBytes, &tmV, bar_addr(ctl.v_full[vs]), bx * 64, U.hk,
                             i * BN, U.b);
          ++gv;
          return true;
        };
        if (!(ok = load_kv(0))) break;
        if (uc > 0 && !(ok = wait_bar(bar_addr(ctl.q_empty), (uc - 1) & 1, ctl, tmo))) break;
        const int nq = U.active1 ? 2 : 1;
        ptx::mbar_arrive_expect_tx(bar_addr(ctl.q_full), (uint32_t)nq * C::TILE);
        for (int i = 0; i < nq; ++i)
          for (int bx = 0; bx < C::NBOX; ++bx)
            ptx::tma_load_4d(sQ + i * C::TILE + bx * kBoxBytes, &tmQ, bar_addr(ctl.q_full), bx * 64, U.head(i),
                             U.row(i), U.b);
        ++uc;
        for (int i = 1; i < U.n_kt && ok; ++i) ok = load_kv(i);
        if (!ok) break;
      }
      if (!ok) {
        // Let every copy already issued land before shared memory is released.
        const unsigned long long drain = 100000000ull;
        if (uc > 0) drain_bar(bar_addr(ctl.q_full), (uc - 1) & 1, drain);
        for (int s = 0; s < KST; ++s)
          if (gk > s) drain_bar(bar_addr(ctl.k_full[s]), ((gk - 1 - s) / KST) & 1, drain);
        for (int s = 0; s < VST; ++s)
          if (gv > s) drain_bar(bar_addr(ctl.v_full[s]), ((gv - 1 - s) / VST) & 1, drain);
      }
    } else if (!skip && warp == 1 && (!(ROTATE && ROT_K) || lane == 0)) {
      // ================================ MMA issuer ============================================
      // Descriptors are built once per operand tile; consecutive K-steps only add a constant to the
      // start-address field (offsets stay inside the 14-bit field), so nothing but an add separates
      // two tcgen05.mma issues.
      using I = Issue<!(ROTATE && ROT_K)>;
      auto issue_S = [&](int iq, uint32_t kbase) {
        const uint64_t dq = ptx::sdesc_sw128(sQ + iq * C::TILE, 16, 1024);
        const uint64_t dk = ptx::sdesc_sw128(kbase, 16, 1024);
        const uint32_t dst = tmem + iq * BN;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t step = (uint64_t)((kk / 4) * (kBoxBytes >> 4) + (kk % 4) * 2);
          I::ss(dst, dq + step, dk + step, IDESC_S, kk > 0 ? 1u : 0u);
        }
      };
      auto issue_PV = [&](int iq, uint32_t vbase, bool first) {
        const uint64_t dv = ptx::sdesc_sw128(vbase, kBoxBytes, 1024);
        const uint32_t dst = tmem + C::COL_O + iq * D, asrc = tmem + iq * BN;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          I::ts(dst, asrc + kk * 8, dv + (uint64_t)(kk * (2048 >> 4)), IDESC_PV, (!first || kk > 0) ? 1u : 0u);
      };
      // Order per key tile i: S0_i, PV1 of the previous q1 step (possibly the previous unit's last),
      // S1_i, PV0_i.  The q1 product of a tile is issued one tile later, so both softmax warpgroups
      // overlap the other tile's products, also across unit boundaries.
      int gk = 0, gv = 0, gp0 = 0, gp1 = 0, uc = 0;
      bool ok = true;
      bool pend = false, pend_vwait = false, pend_first = false, pend_last = false;
      int pend_vs = 0, pend_vph = 0;
      auto flush_pv1 = [&]() -> bool {
        if (!I::wait(bar_addr(ctl.p_full[1]), gp1 & 1, ctl, tmo)) return false;
        if (pend_vwait && !I::wait(bar_addr(ctl.v_full[pend_vs]), pend_vph, ctl, tmo)) return false;
        ptx::tc_fence_after();
        issue_PV(1, sV + pend_vs * C::TILE, pend_first);
        I::commit(bar_addr(ctl.v_empty[pend_vs]));
        if (pend_last) I::commit(bar_addr(ctl.o_full[1]));
        ++gp1;
        pend = false;
        return true;
      };
      FOR_EACH_UNIT(U) {
        // With rotation each query tile has its own ready barrier (S0 may start before q1 is rotated).
        if (!(ok = I::wait(bar_addr(ROTATE ? ctl.q_ready[0] : ctl.q_full), uc & 1, ctl, tmo))) break;
        const uint32_t q1_parity = uc & 1;
        ++uc;
        ptx::tc_fence_after();
        for (int i = 0; i < U.n_kt && ok; ++i) {
          const int ks = gk % KST, kph = (gk / KST) & 1;
          if (!(ok = I::wait(bar_addr(ROTATE && ROT_K ? ctl.k_ready[ks] : ctl.k_full[ks]), kph, ctl, tmo))) break;
          ptx::tc_fence_after();
          const uint32_t kbase = sK + ks * C::TILE;
          const int vs = gv % VST, vph = (gv / VST) & 1;
          if (i < U.n0) {
            issue_S(0, kbase);
            I::commit(bar_addr(ctl.s_full[0]));
          }
          if (pend && !(ok = flush_pv1())) break;
          if (ROTATE && i == 0) {
            if (!(ok = I::wait(bar_addr(ctl.q_ready[1]), q1_parity, ctl, tmo))) break;
            ptx::tc_fence_after();
          }
          if (i < U.n1) {
            issue_S(1, kbase);
            I::commit(bar_addr(ctl.s_full[1]));
          }
          if (i == U.n_kt - 1) I::commit(bar_addr(ctl.q_empty));  // all of this unit's QK^T done
          I::commit(bar_addr(ctl.k_empty[ks]));
          ++gk;
          if (i < U.n0) {
            if (!(ok = I::wait(bar_addr(ctl.p_full[0]), gp0 & 1, ctl, tmo))) break;
            if (!(ok = I::wait(bar_addr(ctl.v_full[vs]), vph, ctl, tmo))) break;
            ptx::tc_fence_after();
            issue_PV(0, sV + vs * C::TILE, i == 0);
            if (U.n1 == 0) I::commit(bar_addr(ctl.v_empty[vs]));
            if (i == U.n0 - 1) I::commit(bar_addr(ctl.o_full[0]));
            ++gp0;
          }
          if (i < U.n1) {
            pend = true;
            pend_vs = vs;
            pend_vph = vph;
            pend_vwait = i >= U.n0;  // V_i not yet seen complete when no PV0 used it
            pend_first = i == 0;
            pend_last = i == U.n1 - 1;
          }
          ++gv;
        }
        if (!ok) break;
      }
      if (ok && pend) ok = flush_pv1();
      // Every MMA issued must finish before tensor memory is freed.
      I::commit(bar_addr(ctl.mma_done));
      drain_bar(bar_addr(ctl.mma_done), 0, 100000000ull);
    }
  } else if (warp < 12) {
    ptx::setmaxnreg_inc<Regs<D, ROTATE>::kSoftmax>();
    if (!skip) {
      // ================================ softmax + epilogue ====================================
      const int wi = (warp - 4) / 4;  // which query tile
      const int r = (warp & 3) * 32 + lane;  // row inside the tile = TMEM lane
      const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
      const uint32_t tS = tmem + lane_off + wi * BN;
      const uint32_t tO = tmem + lane_off + C::COL_O + wi * D;
      const float sl2 = p.scale_log2;
      int gs = 0, uo = 0, uq = 0;
      bool ok = true;
      // Fused: this warpgroup rotates its own query tile of every unit once the tile has landed --
      // a CTA's first unit's at once, each next unit's right after this unit's last softmax step
      // (before the epilogue: the next unit's first O += P V waits for that anyway) -- while the
      // rotation warps turn K tiles; each query tile has its own ready barrier.  cos/sin walk along
      // the thread's rows from the exact value at its first row.
      auto rotate_own_q = [&](int u) -> bool {
        if (!wait_bar_warp(bar_addr(ctl.q_full), uq & 1, ctl, tmo)) return false;
        ++uq;
        const Unit V = decode_unit<VARIANT>(u, p);
        if (wi == 0 || V.active1) {
          int ck, r0;
          rot_mapping<D>((warp & 3) * 32 + lane, ck, r0);
          RopeCS8 step, qcs;
          rope_cs8_exact((uint32_t)RotGeom<D>::RS, sfreq, sfreq + 64, ck * 8, step);
          // Query row i sits at position q_off + i.  Calls with q_off != 0 run the VARIANT kernel.
          int qpos0 = V.row(wi) + r0;
          if constexpr (VARIANT) qpos0 += *reinterpret_cast<volatile int*>(&ctl.q_off);
          rope_cs8_exact((uint32_t)qpos0, sfreq, sfreq + 64, ck * 8, qcs);
          if constexpr (VARIANT)
            rotate_tile_variant<D, BF16>(sQ + wi * C::TILE, r0, ck, qcs, step, p.rot_chunks, p.interleaved != 0,
                                         p.qpos ? p.qpos + (size_t)V.b * p.N + V.row(wi) : nullptr,
                                         p.N - V.row(wi), sfreq);
          else
            rotate_tile<D, BF16>(sQ + wi * C::TILE, r0, ck, qcs, step);
          ptx::fence_proxy_async_smem();
        }
        ptx::mbar_arrive(bar_addr(ctl.q_ready[wi]));
        return true;
      };
      if constexpr (ROTATE && ROT_K) {
        const int u0 = unit_at(0, p);
        if (u0 >= 0) ok = rotate_own_q(u0);
      }
      for (int k = 0, u; ok && (u = unit_at(k, p)) >= 0; ++k) {
        const Unit U = decode_unit<VARIANT>(u, p);
        const int n_steps = wi == 0 ? U.n0 : U.n1;  // 0: an inactive q1 (its key loop and epilogue skipped)
        const int qt = U.row(wi) / BM;
        // Key column c of tile j is visible to row r iff c <= q_off + qt*128 + r - j*128; tiles
        // j >= j_mask have that limit below 127 for some row and take the per-element mask (the
        // diagonal tile, and the one after it when q_off is not a multiple of 128).  Without extra
        // keys (VARIANT = false: q_off = 0) that is the last tile, j = qt, with limit r.
        const int j_mask = VARIANT ? (p.q_off + qt * BM + 1) / BN : n_steps - 1;
        float m_run = -INFINITY, l_run = 0.f;
        for (int j = 0; j < n_steps && ok; ++j) {
          if (!(ok = wait_bar_warp(bar_addr(ctl.s_full[wi]), gs & 1, ctl, tmo))) break;
          ++gs;
          ptx::tc_fence_after();
          const bool diag = j >= j_mask;
          const int lim = VARIANT ? p.q_off + (qt - j) * BM + r : r;
          uint32_t sv[4][32];
#pragma unroll
          for (int c = 0; c < 4; ++c) ptx::tmem_ld32(tS + 32 * c, sv[c]);
          ptx::tmem_wait_ld();
          if (diag) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (32 * c + e > lim) sv[c][e] = __float_as_uint(-INFINITY);
          }
          if (j == 0) m_run = row_max128(sv) * sl2;  // the first tile of a row sets the max
          // P with the running max, kept in registers until the row sums pass the check (S stays
          // intact in tensor memory until then).
          uint32_t pk[64];
          float sum = softmax_p<BF16>(sv, sl2, m_run, pk);
          const bool need = !(sum <= kSumCap);  // also catches inf / nan
          if (__any_sync(0xFFFFFFFFu, need)) {
            const RowState st = softmax_redo<D, BF16>(tS, tO, lim, diag, need, sl2, m_run, l_run);
            sum = st.sum;
            m_run = st.m;
            l_run = st.l;
          } else {
#pragma unroll
            for (int c = 0; c < 4; ++c)
              ptx::tmem_st16(tS + 16 * c, *reinterpret_cast<const uint32_t(*)[16]>(&pk[16 * c]));
          }
          l_run += sum;
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar_addr(ctl.p_full[wi]));
        }
        if (!ok) break;
        if constexpr (ROTATE && ROT_K) {
          const int un = unit_at(k + 1, p);
          if (un >= 0 && !(ok = rotate_own_q(un))) break;
        }
        if (n_steps == 0) continue;
        if (!(ok = wait_bar_warp(bar_addr(ctl.o_full[wi]), uo & 1, ctl, tmo))) break;
        ++uo;
        ptx::tc_fence_after();
        const int row = qt * BM + r;
        const float inv_l = 1.f / l_run;
        const int head = U.head(wi);
        T* orow = reinterpret_cast<T*>(p.out) + (((size_t)U.b * p.N + row) * p.Hq + head) * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          ptx::tmem_ld32(tO + 32 * c, o);
          ptx::tmem_wait_ld();
          uint32_t w[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            w[e] = Pack<BF16>::pack(__uint_as_float(o[2 * e]) * inv_l, __uint_as_float(o[2 * e + 1]) * inv_l);
          if (row < p.N) {
            uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
            for (int v = 0; v < 4; ++v) dst[v] = make_uint4(w[4 * v], w[4 * v + 1], w[4 * v + 2], w[4 * v + 3]);
          }
        }
        if (row < p.N && p.lse != nullptr)
          p.lse[((size_t)U.b * p.Hq + head) * p.N + row] = (m_run + log2f(l_run)) * kLn2;
        // The O reads above completed (wait::ld) before this warpgroup's next p_full arrive, which
        // is what lets the next unit's first O += P V overwrite O.
      }
    }
  } else {
    ptx::setmaxnreg_dec<Regs<D, ROTATE>::kRotate>();
    if constexpr (ROTATE) {
      if (!skip) {
        // ================================ K tile rotation =======================================
        // cos/sin are carried along the thread's rows by angle addition with the exact rotation of
        // RS rows, exact at the first row of every 16th key tile (one fp32 rounding per step, at most
        // 128 steps between exact values: relative drift < 1e-5).  Fused: the query tiles are
        // rotated by the softmax warpgroups.  Split: K arrives rotated (the pre-rotation pass) and
        // these warps rotate the query tiles instead, each arriving on its own ready barrier.
        if constexpr (!ROT_K) {
          int ck, r0;
          rot_mapping<D>(threadIdx.x - 384, ck, r0);
          RopeCS8 step;
          rope_cs8_exact((uint32_t)RotGeom<D>::RS, sfreq, sfreq + 64, ck * 8, step);
          int uc = 0;
          FOR_EACH_UNIT(U) {
            if (!wait_bar_warp(bar_addr(ctl.q_full), uc & 1, ctl, tmo)) break;
            ++uc;
            for (int tq = 0; tq < 2; ++tq) {
              if (tq == 0 || U.active1) {
                RopeCS8 qcs;
                int qpos0 = U.row(tq) + r0;
                if constexpr (VARIANT) qpos0 += *reinterpret_cast<volatile int*>(&ctl.q_off);
                rope_cs8_exact((uint32_t)qpos0, sfreq, sfreq + 64, ck * 8, qcs);
                if constexpr (VARIANT)
                  rotate_tile_variant<D, BF16>(sQ + tq * C::TILE, r0, ck, qcs, step, p.rot_chunks,
                                               p.interleaved != 0,
                                               p.qpos ? p.qpos + (size_t)U.b * p.N + U.row(tq) : nullptr,
                                               p.N - U.row(tq), sfreq);
                else
                  rotate_tile<D, BF16>(sQ + tq * C::TILE, r0, ck, qcs, step);
                ptx::fence_proxy_async_smem();
              }
              ptx::mbar_arrive(bar_addr(ctl.q_ready[tq]));
            }
          }
        }
        if constexpr (ROT_K) {
          constexpr int kReseed = 16;
          int ck, r0;
          rot_mapping<D>(threadIdx.x - 384, ck, r0);
          RopeCS8 step;
          rope_cs8_exact((uint32_t)RotGeom<D>::RS, sfreq, sfreq + 64, ck * 8, step);
          int gk = 0;
          bool ok = true;
          FOR_EACH_UNIT(U) {
            RopeCS8 kcs;
            for (int i = 0; i < U.n_kt && ok; ++i) {
              if (i % kReseed == 0) rope_cs8_exact((uint32_t)(i * BN + r0), sfreq, sfreq + 64, ck * 8, kcs);
              const int ks = gk % KST, kph = (gk / KST) & 1;
              if (!(ok = wait_bar_warp(bar_addr(ctl.k_full[ks]), kph, ctl, tmo))) break;
              ++gk;
              // Half-split over all d entries: the tuned path; other RoPE forms (VARIANT kernels) take
              // rotate_tile_variant.
              if constexpr (VARIANT)
                rotate_tile_variant<D, BF16>(sK + ks * C::TILE, r0, ck, kcs, step, p.rot_chunks, p.interleaved != 0,
                                             p.kpos ? p.kpos + (size_t)U.b * p.Nk + i * BN : nullptr, p.Nk - i * BN,
                                             sfreq);
              else
                rotate_tile<D, BF16>(sK + ks * C::TILE, r0, ck, kcs, step);
              ptx::fence_proxy_async_smem();
              ptx::mbar_arrive(bar_addr(ctl.k_ready[ks]));
            }
            if (!ok) break;
          }
        }
      }
    }
  }

  // ---- teardown: every role reaches here; no tcgen05 work is in flight --------------------
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

// One CTA of 32 threads that waits on a barrier no one arrives on, for at most timeout_ns.
__global__ void diag_wait_timeout_kernel(unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    ptx::mbar_init(ptx::smem_u32(&bar), 1);
    ptx::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint64_t t0 = ptx::globaltimer_ns();
    for (;;) {
      if (ptx::mbar_try_wait(ptx::smem_u32(&bar), 0)) break;  // never true: nothing arrives
      if (ptx::globaltimer_ns() - t0 > timeout_ns) {
        atomicOr(&g_device_status, 1u);
        break;
      }
    }
  }
  __syncthreads();
}

template <int D, bool ROTATE, bool BF16, bool VARIANT, bool ROT_K>
cudaError_t launch_one(const AttnMaps& maps, const AttnParams& p, cudaStream_t stream, const char** why) {
  auto kernel = attn_fwd_kernel<D, ROTATE, BF16, VARIANT, ROT_K>;
  static DeviceOnce once;  // per instantiation: attributes set and SM count kept per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  bool regs_ok = true;
  int sms = 0;
  e = once.get(dev, [&](int* out) -> cudaError_t {
    cudaError_t r = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg<D>::SMEM);
    if (r != cudaSuccess) return r;
    cudaFuncAttributes attr;
    r = cudaFuncGetAttributes(&attr, kernel);
    if (r != cudaSuccess) return r;
    // The warp-role register split (setmaxnreg) hands out exactly 512 x 128 registers: launching
    // with fewer per thread would leave the softmax warps waiting for registers forever.
    if (attr.numRegs != 128) {
      regs_ok = false;
      return cudaErrorInvalidConfiguration;
    }
    return cudaDeviceGetAttribute(out, cudaDevAttrMultiProcessorCount, dev);
  }, &sms);
  if (e != cudaSuccess) {
    if (!regs_ok && why) *why = "attention kernel was not compiled with 128 registers per thread (setmaxnreg split)";
    return e;
  }
  // Persistent: one CTA per SM (shared memory and registers admit only one), each walking its share
  // of the work units.
  const int grid = p.total_units < sms ? p.total_units : sms;
  // After this library's pre-rotation pass the kernel is launched as a programmatic dependent: its
  // prologue (barriers, tensor memory, descriptor prefetch) overlaps the end of the pass, and the
  // TMA producer waits for the pass before its first load.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg<D>::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.after_rope_pass ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kernel, maps.q, maps.k, maps.v, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Rotation mode r: 0 none (pre-rotated Q and K), 1 Q and K (fused), 2 Q only (split: K pre-rotated).
template <int D, bool BF16, bool VARIANT>
cudaError_t launch_mode(const AttnMaps& maps, const AttnParams& p, int r, cudaStream_t stream, const char** why) {
  if (r == 1) return launch_one<D, true, BF16, VARIANT, true>(maps, p, stream, why);
  if (r == 2) return launch_one<D, true, BF16, VARIANT, false>(maps, p, stream, why);
  return launch_one<D, false, BF16, VARIANT, false>(maps, p, stream, why);
}

template <int D>
cudaError_t launch_d(const AttnMaps& maps, const AttnParams& p, bool bf16, bool variant, int r, cudaStream_t stream,
                     const char** why) {
  if (variant)
    return bf16 ? launch_mode<D, true, true>(maps, p, r, stream, why) : launch_mode<D, false, true>(maps, p, r, stream, why);
  return bf16 ? launch_mode<D, true, false>(maps, p, r, stream, why) : launch_mode<D, false, false>(maps, p, r, stream, why);
}

}  // namespace

cudaError_t launch_attn_fwd(const AttnMaps& maps, const AttnParams& p, int d, bool bf16, bool rotate_q,
                            bool rotate_k, cudaStream_t stream, const char** why) {
  if (p.total_units <= 0) return cudaSuccess;
  // The default kernels handle N == Nk and the half-split form over all d entries at positions i
  // and j; every other case takes the VARIANT instantiation.
  const bool variant = p.q_off != 0 || (rotate_q && (!(p.rot_chunks == d / 16 && p.interleaved == 0) ||
                                                     p.qpos != nullptr || p.kpos != nullptr));
  const int r = !rotate_q ? 0 : (rotate_k ? 1 : 2);
  return d == 128 ? launch_d<128>(maps, p, bf16, variant, r, stream, why)
                  : launch_d<64>(maps, p, bf16, variant, r, stream, why);
}

cudaError_t read_and_clear_device_status(unsigned int* value, cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(value, g_device_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  if (*value != 0u) {
    const unsigned int zero = 0u;
    e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(unsigned int));
  }
  return e;
}

cudaError_t launch_diag_wait_timeout(unsigned long long timeout_ns, cudaStream_t stream) {
  diag_wait_timeout_kernel<<<1, 32, 0, stream>>>(timeout_ns);
  return cudaGetLastError();
}

}  // namespace attnfuse
