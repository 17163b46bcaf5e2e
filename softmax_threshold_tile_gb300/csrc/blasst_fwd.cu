// Skip-Softmax (BLASST) attention forward for GB300 (sm_103a).
//
// The method ("Skip-Softmax" design doc, vLLM-Omni, section "Algorithm"; the
// same doc on docs.vllm.ai, sections "The online-softmax pass" and "The skip
// test"): FlashAttention's streaming online-softmax pass over key tiles of 128.
// Tile scores S_j = Q K_j^T * scale are always computed; when every query row i
// of the 128-row query tile has tile_max[i] - running_max[i] < ln(lambda), the
// tile's exponentials, its l / O update and its P V product are skipped.
// lambda = factor / Sk ("From configuration to the kernel threshold").
//
// One CTA owns two 128-row query tiles (A and B) of one (batch, head) and streams
// every key tile once for both through a warp-specialised pipeline:
//   warps 0-7  softmax, all eight on one tile at a time (A, then B, for every key
//              tile): warps w and w + 4 share the TMEM lanes of rows 32 (w % 4) ...
//              + 31 and take key columns 0-63 and 64-127. tcgen05.ld of S_j, half-row
//              max, an AND-vote of the skip test over the tile's 128 rows (named
//              barrier, which also publishes the half-row maxima), exp2 of a kept
//              tile written back into TMEM as bf16 P (over S_j), conditional O
//              rescale, epilogue (O / l -> bf16, lse).
//   warp 8     MMA: the whole warp runs the issue loop and one elected lane issues
//              tcgen05.mma, alternating the two tiles so that one tile's softmax
//              overlaps the other tile's matrix work:
//                O_A += P_A(j) V_j ; S_A = Q_A K_{j+1}^T ; O_B += P_B(j) V_j ; S_B = Q_B K_{j+1}^T
//              P V is issued only for a tile that kept key tile j.
//   warp 9     TMA producer: both Q tiles once, K tiles one ahead through a 2-stage ring,
//              and V_j only once a tile has kept key tile j (as soon as tile A keeps it,
//              otherwise after tile B's decision): a key tile both tiles skip is never loaded.
// TMEM (512 columns): S_A [0,128), S_B [128,256), O_A [256,384), O_B [384,512).
// Shared memory: Q_A, Q_B, 2 x K, 2 x V tiles of 32 KiB, all 128-byte swizzled.
//
// Numerics: scores are fp32 from bf16 operands; the test is evaluated in log2
// units, (tile_max - running_max) * scale * log2(e) < log2(lambda), which is the
// design doc's log-space test scaled by log2(e). P is rounded to bf16 for P V; l and O
// accumulate in fp32. The exponent reference m_use trails the true running max
// by at most 8 (log2 units), so O is rescaled only when the max grows by more
// than that; the skip test always uses the true running max.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstddef>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "blasst.h"
#include "blasst_internal.h"
#include "sm103_ptx.cuh"

namespace blasst {
namespace {

using namespace ptx;

constexpr int kTile = 128;      // query rows per query tile == keys per key tile
constexpr int kHeadDim = 128;   // d
constexpr int kQTiles = 2;      // query tiles per CTA
constexpr int kSoftmaxWarps = 4;             // warps that cover the 128 TMEM lanes once
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;  // the softmax runs kQTiles x this many threads
constexpr int kMmaWarp = kQTiles * kSoftmaxWarps;   // 8
constexpr int kLoadWarp = kMmaWarp + 1;             // 9
constexpr int kThreads = 3 * 128;                   // 384: two softmax warpgroups + one for MMA / TMA
// Register budget: 384 threads launch with 168 registers each (64512 in all); the two softmax
// warpgroups grow to 224 and the MMA / TMA warpgroup shrinks to 56:
// 2 x 128 x 224 + 128 x 56 = 64512.
constexpr uint32_t kSoftmaxRegs = 224;
constexpr uint32_t kControlRegs = 56;
static_assert(2 * 128 * kSoftmaxRegs + 128 * kControlRegs <= kThreads * 168, "register split");
constexpr int kStages = 2;
constexpr uint32_t kTileBytes = kTile * kHeadDim * 2;  // one bf16 128 x 128 tile
constexpr uint32_t kTileBytesF8 = kTile * kHeadDim;    // one e4m3 128 x 128 tile (128-B rows)
constexpr uint32_t kHalfBytes = kTileBytes / 2;        // 128 rows x 64 features (128-B rows)
constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr uint32_t col_s(int t) { return static_cast<uint32_t>(t) * 128u; }
__host__ __device__ constexpr uint32_t col_o(int t) { return 256u + static_cast<uint32_t>(t) * 128u; }
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2 = 0.693147180559945309f;
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // a single wait may last at most 2 s
constexpr uint64_t kDrainTimeoutNs = 50000000ull;   // waits for in-flight copies / MMAs at exit

// Bits of the device error word: which role gave up waiting.
constexpr uint32_t kErrProducer = 1u << 0;
constexpr uint32_t kErrMma = 1u << 1;
constexpr uint32_t kErrSoftmax = 1u << 2;
constexpr uint32_t kErrDrain = 1u << 3;
constexpr uint32_t kErrGeometry = 1u << 4;  // packed-document offsets out of order or too long

__device__ uint32_t g_error_word;

struct alignas(1024) Smem {
  uint8_t q[kQTiles][kTileBytes];
  uint8_t k[kStages][kTileBytes];
  uint8_t v[kStages][kTileBytes];
  uint64_t q_full;
  uint64_t k_full[kStages];
  uint64_t v_full[kStages];
  uint64_t s_full[kQTiles];   // S of tile t for key tile j is in TMEM (tcgen05.commit, phase j)
  uint64_t dec[kQTiles][2];   // tile t has decided key tile j (slot j % 2); flag in skip_flag
  uint64_t p_ready[kQTiles];  // softmax t is done with S: decision taken, P written, O rescaled
  uint64_t o_done[kQTiles];   // every MMA of the CTA has completed (one phase, after the loop)
  uint64_t drain;             // all MMAs of the CTA have completed
  uint32_t tmem_base;
  uint32_t skip_flag[kQTiles][2];  // decision of tile t on key tile j, slot j % 2
  uint32_t quit[kQTiles][2];  // the softmax warps leave the loop together (tile, step parity)
  float hmax[kQTiles][2][kTile];   // half-row maxima of the current key tile (tile, half, row)
  float lpart[kQTiles][2][kTile];  // half-row sums at the end (tile, half, row)
  uint32_t abort;             // non-zero once some role gave up waiting: the roles' error bits
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;  // + slack to align the base to 1024 B

struct FwdParams {
  int B, H, Sq, Sk, nQ, nK;  // fixed-length batch; in varlen mode Sq / Sk are the maxima
  float scale_log2;   // scale (times both descales for e4m3 Q / K) * log2(e)
  float log2_lambda;  // log2(factor / Sk); -inf when factor == 0
  __nv_bfloat16* o;
  float* lse;
  float* max_prob;
  uint32_t* skip_counts;
  uint8_t* skip_mask;
  const int* cu_q;    // varlen: token offsets of the B documents (B + 1 values), else null
  const int* cu_k;
  int Tq, Tk;         // varlen: total query / key tokens (token extents of the packed tensors)
  int min_seq_len;    // documents with fewer keys than this run dense
  int withhold_k;     // test of the bounded waits: the copy of this key tile is never issued (-1: off)
  uint32_t* status;   // the caller's device status word, or null
};

// Error bits go to the device-wide word and, when the caller passed one, to its status word.
__device__ __forceinline__ void report_error(uint32_t* status, uint32_t bits) {
  atomicOr(&g_error_word, bits);
  if (status) atomicOr(status, bits);
}

// What one CTA works on: one batch entry (or packed document) and head, and its lengths.
struct Geo {
  int Sq, Sk;          // query / key length of this entry
  int nQ, nK;          // its query / key tiles
  int q_tok0, k_tok0;  // its first token in the token dimension of the TMA views
  int tma_b;           // its batch coordinate in the TMA views (0 for packed documents)
  float log2_lambda;
};

// Output addresses of token s of the CTA's entry (computed in the epilogue, not held live):
// o row (o_tok0 + s) * H + h, lse / max_prob index stat0 + s.
template <bool kVarlen>
__device__ __forceinline__ size_t out_tok0(const FwdParams& p, const Geo& g, int b) {
  return kVarlen ? static_cast<size_t>(g.q_tok0) : static_cast<size_t>(b) * p.Sq;
}
template <bool kVarlen>
__device__ __forceinline__ size_t stat_base(const FwdParams& p, const Geo& g, int b, int h) {
  return kVarlen ? static_cast<size_t>(h) * p.Tq + g.q_tok0 : (static_cast<size_t>(b) * p.H + h) * p.Sq;
}

// The lengths and threshold the hot loops read: straight from the kernel parameters for a
// fixed-length batch (constant-bank operands, no registers held), from the CTA's geometry
// for packed documents.
template <bool kVarlen>
struct Lens {
  const FwdParams& p;
  const Geo& g;
  __device__ __forceinline__ int nK() const { return kVarlen ? g.nK : p.nK; }
  __device__ __forceinline__ int Sk() const { return kVarlen ? g.Sk : p.Sk; }
  __device__ __forceinline__ float log2_lambda() const { return kVarlen ? g.log2_lambda : p.log2_lambda; }
  __device__ __forceinline__ int k_tok0() const { return kVarlen ? g.k_tok0 : 0; }
};

// Fixed-length batches take every length from the kernel parameters; packed documents read
// their offset tables.
template <bool kVarlen>
__device__ __forceinline__ Geo make_geo(const FwdParams& p, int b, int h) {
  Geo g;
  if (kVarlen) {
    // Offsets come from the caller's device memory: clamp them into the packed tensors so
    // that a bad table can never address outside them, and report it.
    const int q0 = p.cu_q[b], q1 = p.cu_q[b + 1], k0 = p.cu_k[b], k1 = p.cu_k[b + 1];
    g.q_tok0 = min(max(q0, 0), p.Tq);
    g.k_tok0 = min(max(k0, 0), p.Tk);
    g.Sq = min(max(q1, g.q_tok0), p.Tq) - g.q_tok0;
    g.Sk = min(max(k1, g.k_tok0), p.Tk) - g.k_tok0;
    if (q0 < 0 || k0 < 0 || q1 < q0 || k1 < k0 || q1 > p.Tq || k1 > p.Tk || g.Sq > p.Sq || g.Sk > p.Sk) {
      if (threadIdx.x == 0 && blockIdx.x == 0 && blockIdx.y == 0) report_error(p.status, kErrGeometry);
      g.Sq = min(g.Sq, p.Sq);
      g.Sk = min(g.Sk, p.Sk);
    }
    g.tma_b = 0;
  } else {
    g.q_tok0 = 0;
    g.k_tok0 = 0;
    g.Sq = p.Sq;
    g.Sk = p.Sk;
    g.tma_b = b;
  }
  if (kVarlen) {
    g.nQ = (g.Sq + kTile - 1) / kTile;
    g.nK = (g.Sk + kTile - 1) / kTile;
    // Short documents run dense (the per-document dense fallback of packed batches).
    g.log2_lambda = g.Sk < p.min_seq_len ? -INFINITY : p.log2_lambda;
  } else {
    g.nQ = p.nQ;
    g.nK = p.nK;
    g.log2_lambda = p.log2_lambda;  // the host applies min_seq_len to the one length
  }
  return g;
}

// Bounded wait on an mbarrier phase. Gives up after `timeout_ns`, or at once when
// another role has given up (unless `respect_abort` is false); on a timeout it ORs `site` into
// the CTA's abort word, which the CTA reports device-wide (and to the caller's status word) when
// it ends.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile uint32_t* abort,
                                         uint32_t site, bool respect_abort = true,
                                         uint64_t timeout_ns = kWaitTimeoutNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((n & 15u) == 0) {
      if (respect_abort && *abort) return false;
      if (globaltimer_ns() - t0 > timeout_ns) {
        atomicOr(const_cast<uint32_t*>(abort), site);  // reported when the CTA ends
        return false;
      }
    }
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  uint32_t u;
  memcpy(&u, &v, sizeof u);
  return u;
}

// ------------------------------------------------------------------ producer
template <bool kVarlen, bool kFp8>
__device__ __forceinline__ void run_producer(Smem& sm, const CUtensorMap* tq, const CUtensorMap* tk,
                                             const CUtensorMap* tv, const FwdParams& p, const Geo& g, int h,
                                             int qt0) {
  const Lens<kVarlen> L{p, g};
  volatile uint32_t* abort = &sm.abort;
  prefetch_tmap(tq);
  prefetch_tmap(tk);
  prefetch_tmap(tv);
  const uint32_t q_full = smem_u32(&sm.q_full);
  // e4m3 Q / K tiles are one box of 128 rows x 128 B; bf16 tiles two boxes of 64 features.
  constexpr uint32_t kQKBytes = kFp8 ? kTileBytesF8 : kTileBytes;
  mbar_arrive_expect_tx(q_full, kQTiles * kQKBytes);
#pragma unroll
  for (int t = 0; t < kQTiles; ++t) {
    const uint32_t qs = smem_u32(sm.q[t]);
    tma_load_4d(qs, tq, q_full, 0, h, g.q_tok0 + (qt0 + t) * kTile, g.tma_b);
    if (!kFp8) tma_load_4d(qs + kHalfBytes, tq, q_full, 64, h, g.q_tok0 + (qt0 + t) * kTile, g.tma_b);
  }

  // Copy n goes to stage n % 2, over copy n - 2. No "stage empty" barrier is needed: both
  // tiles' decisions on key tile i are published only after their softmax has read S(i), and
  // S_B(i) is committed after every earlier MMA of the CTA. So once this thread has waited for
  // both decisions on key tile i, every MMA up to Q_B K_i^T has completed, which covers the
  // readers of K_(i) and of every V tile used before key tile i. K_(j+1) is issued after the
  // decisions on key tile j - 1 (its stage held K_(j-1)); V copy n, at key tile j, after the
  // decisions on key tile j - 1, while copy n - 2 served a key tile at most j - 2.
  int k_issued = 0, v_issued = 0;
  auto issue_k = [&](int j) {
    const int st = k_issued & 1;
    if (j == p.withhold_k) {  // the waits on this copy run out (see launch())
      ++k_issued;
      return;
    }
    const uint32_t kf = smem_u32(&sm.k_full[st]);
    const uint32_t ks = smem_u32(sm.k[st]);
    mbar_arrive_expect_tx(kf, kQKBytes);
    tma_load_4d(ks, tk, kf, 0, h, L.k_tok0() + j * kTile, g.tma_b);
    if (!kFp8) tma_load_4d(ks + kHalfBytes, tk, kf, 64, h, L.k_tok0() + j * kTile, g.tma_b);
    ++k_issued;
  };
  auto issue_v = [&](int j) {
    const int st = v_issued & 1;
    const uint32_t vf = smem_u32(&sm.v_full[st]);
    const uint32_t vs = smem_u32(sm.v[st]);
    mbar_arrive_expect_tx(vf, kTileBytes);
    tma_load_4d(vs, tv, vf, 0, h, L.k_tok0() + j * kTile, g.tma_b);
    tma_load_4d(vs + kHalfBytes, tv, vf, 64, h, L.k_tok0() + j * kTile, g.tma_b);
    ++v_issued;
  };
  issue_k(0);
  bool ok = true;
  for (int j = 0; j < L.nK() && ok; ++j) {
    if (j + 1 < L.nK()) issue_k(j + 1);
    // V_j is needed if either tile keeps key tile j. Both decisions are waited for on every
    // j, so each decision barrier slot is waited once per use and its parity cannot alias (a
    // tile can decide key tile j + 1 at most before this wait, never j + 2).
    bool loaded = false;
#pragma unroll
    for (int t = 0; t < kQTiles; ++t) {
      if (!wait_bar(smem_u32(&sm.dec[t][j & 1]), (j >> 1) & 1, abort, kErrProducer)) { ok = false; break; }
      const uint32_t skip = *reinterpret_cast<volatile uint32_t*>(&sm.skip_flag[t][j & 1]);
      if (!skip && !loaded) {
        issue_v(j);
        loaded = true;
      }
    }
  }
  // Copy n went to stage n % 2 as that stage's (n / 2)-th use, completing phase parity (n / 2) & 1.
#pragma unroll
  for (int back = 1; back <= kStages; ++back) {
    const int nk = k_issued - back, nv = v_issued - back;
    if (nk >= 0)
      wait_bar(smem_u32(&sm.k_full[nk & 1]), (nk >> 1) & 1, abort, kErrDrain, false, kDrainTimeoutNs);
    if (nv >= 0)
      wait_bar(smem_u32(&sm.v_full[nv & 1]), (nv >> 1) & 1, abort, kErrDrain, false, kDrainTimeoutNs);
  }
  wait_bar(q_full, 0, abort, kErrDrain, false, kDrainTimeoutNs);
}

// ------------------------------------------------------------------ MMA issuer
// Every lane of a converged warp waits; the result is the same in every lane.
__device__ __forceinline__ bool wait_bar_w(uint32_t bar, uint32_t parity, volatile uint32_t* abort,
                                           uint32_t site, bool respect_abort = true,
                                           uint64_t timeout_ns = kWaitTimeoutNs) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, abort, site, respect_abort, timeout_ns));
}

// Run by all 32 lanes of the MMA warp. Waits and flag reads give every lane the same result, so
// the warp stays converged, and one elected lane (always lane 0) issues the MMAs and commits.
template <bool kVarlen, bool kFp8>
__device__ __forceinline__ void run_mma(Smem& sm, uint32_t tmem, const FwdParams& p, const Geo& g) {
  const Lens<kVarlen> L{p, g};
  volatile uint32_t* abort = &sm.abort;
  constexpr uint32_t kIdescQK = kFp8 ? idesc_e4m3_f32(kTile, kTile)          // K tile is K-major
                                     : idesc_bf16_f32(kTile, kTile, false);
  constexpr uint32_t kIdescPV = idesc_bf16_f32(kTile, kHeadDim, true);   // V tile is MN-major

  // Descriptors of every operand tile, built once; a K step only adds (offset >> 4) to the
  // 14-bit start-address field, which never carries out of it (all tiles lie below 256 KiB).
  // (Stage-indexed values are selected, not indexed, so that they stay in registers.)
  const uint64_t dq0 = smem_desc_sw128(smem_u32(sm.q[0]), 16, 1024);
  const uint64_t dq1 = smem_desc_sw128(smem_u32(sm.q[1]), 16, 1024);
  const uint64_t dk0 = smem_desc_sw128(smem_u32(sm.k[0]), 16, 1024);
  const uint64_t dk1 = smem_desc_sw128(smem_u32(sm.k[1]), 16, 1024);
  const uint64_t dv0 = smem_desc_sw128(smem_u32(sm.v[0]), kHalfBytes, 1024);
  const uint64_t dv1 = smem_desc_sw128(smem_u32(sm.v[1]), kHalfBytes, 1024);
  // S_t = Q_t K^T: 8 steps of K = 16 features. Q and K tiles are two 64-feature halves of
  // 128-B swizzled rows; a step advances 32 B inside a half (SBO = 8 rows x 128 B).
  auto issue_qk = [&](int t, int st) {
    const uint64_t aq = t ? dq1 : dq0;
    const uint64_t bk = st ? dk1 : dk0;
    const uint32_t d = tmem + col_s(t);
    if (kFp8) {
      // e4m3: 4 steps of K = 32 features, 32 B apart inside the one 128-B swizzled row.
      mma_ss_f8_off_w<0, 0>(d, aq, bk, kIdescQK, 0u);
      mma_ss_f8_off_w<2, 2>(d, aq, bk, kIdescQK, 1u);
      mma_ss_f8_off_w<4, 4>(d, aq, bk, kIdescQK, 1u);
      mma_ss_f8_off_w<6, 6>(d, aq, bk, kIdescQK, 1u);
      return;
    }
    mma_ss_off_w<0, 0>(d, aq, bk, kIdescQK, 0u);
    mma_ss_off_w<2, 2>(d, aq, bk, kIdescQK, 1u);       // +32 B
    mma_ss_off_w<4, 4>(d, aq, bk, kIdescQK, 1u);       // +64 B
    mma_ss_off_w<6, 6>(d, aq, bk, kIdescQK, 1u);       // +96 B
    mma_ss_off_w<1024, 1024>(d, aq, bk, kIdescQK, 1u); // second 64-feature half (+16 KiB)
    mma_ss_off_w<1026, 1026>(d, aq, bk, kIdescQK, 1u);
    mma_ss_off_w<1028, 1028>(d, aq, bk, kIdescQK, 1u);
    mma_ss_off_w<1030, 1030>(d, aq, bk, kIdescQK, 1u);
  };
  // O_t (+)= P_t V: 8 steps of K = 16 keys. P sits in TMEM over S_t (2 bf16 per column, 8
  // columns per step). V rows are keys: a step advances 16 rows = 2 KiB (128 in the
  // descriptor); the two 64-feature halves are LBO = 16 KiB apart, 8-row groups SBO = 1 KiB.
  auto issue_pv = [&](int t, int st, bool accumulate) {
    const uint64_t bv = st ? dv1 : dv0;
    const uint32_t d = tmem + col_o(t);
    const uint32_t a = tmem + col_s(t);
    mma_ts_off_w<0>(d, a, bv, kIdescPV, accumulate ? 1u : 0u);
    mma_ts_off_w<128>(d, a + 8, bv, kIdescPV, 1u);
    mma_ts_off_w<256>(d, a + 16, bv, kIdescPV, 1u);
    mma_ts_off_w<384>(d, a + 24, bv, kIdescPV, 1u);
    mma_ts_off_w<512>(d, a + 32, bv, kIdescPV, 1u);
    mma_ts_off_w<640>(d, a + 40, bv, kIdescPV, 1u);
    mma_ts_off_w<768>(d, a + 48, bv, kIdescPV, 1u);
    mma_ts_off_w<896>(d, a + 56, bv, kIdescPV, 1u);
  };

  int pv_issued0 = 0, pv_issued1 = 0;
  bool ok = wait_bar_w(smem_u32(&sm.q_full), 0, abort, kErrMma) &&
            wait_bar_w(smem_u32(&sm.k_full[0]), 0, abort, kErrMma);
  if (ok) {
    tc_fence_after();
#pragma unroll
    for (int t = 0; t < kQTiles; ++t) {
      issue_qk(t, 0);
      tc_commit_w(smem_u32(&sm.s_full[t]));
    }
    int v_used = 0;  // V tiles consumed so far; V copy n sits in stage n % 2
    for (int j = 0; j < L.nK() && ok; ++j) {
      const int st = v_used & 1;
      const uint32_t parity = (v_used >> 1) & 1;
      const int nst = (j + 1) & 1;
      const bool has_next = j + 1 < L.nK();
      bool v_ready = false;
      bool any_kept = false;
#pragma unroll
      for (int t = 0; t < kQTiles; ++t) {
        // p_ready arrives once the tile has read S_t and decided: at once for a skipped
        // key tile, after P is written (and O rescaled) for a kept one.
        if (!wait_bar_w(smem_u32(&sm.p_ready[t]), j & 1, abort, kErrMma)) { ok = false; break; }
        tc_fence_after();
        const uint32_t skip = *reinterpret_cast<volatile uint32_t*>(&sm.skip_flag[t][j & 1]);
        if (!skip) {
          if (!v_ready) {
            if (!wait_bar_w(smem_u32(&sm.v_full[st]), parity, abort, kErrMma)) { ok = false; break; }
            tc_fence_after();
            v_ready = true;
          }
          issue_pv(t, st, (t ? pv_issued1 : pv_issued0) > 0);
          if (t) ++pv_issued1; else ++pv_issued0;
          any_kept = true;
        }
        if (has_next) {
          // S_t is free: it was read before p_ready, and its P (if the tile was kept) is
          // read by the P V just issued; tcgen05.mma executes in issue order.
          if (t == 0) {
            if (!wait_bar_w(smem_u32(&sm.k_full[nst]), ((j + 1) >> 1) & 1, abort, kErrMma)) { ok = false; break; }
            tc_fence_after();
          }
          issue_qk(t, nst);
          tc_commit_w(smem_u32(&sm.s_full[t]));
        }
      }
      if (!ok) break;
      if (any_kept) ++v_used;  // V_j was loaded (some tile kept key tile j)
    }
  }
  // The softmax epilogues read O once every P V has completed. Inside the loop no such signal
  // is needed: S_t(j + 1) is committed after the P V of key tile j, and a commit tracks every
  // earlier MMA of this thread, so a softmax that has S_t(j + 1) knows its earlier P V are
  // done. Committed on every exit path, so the epilogue waits never hang.
#pragma unroll
  for (int t = 0; t < kQTiles; ++t) tc_commit_w(smem_u32(&sm.o_done[t]));
  // Every MMA this thread issued completes before TMEM is released.
  tc_commit_w(smem_u32(&sm.drain));
  wait_bar_w(smem_u32(&sm.drain), 0, abort, kErrDrain, false, kDrainTimeoutNs);
}

// ------------------------------------------------------------------ softmax + epilogue
// All eight softmax warps work on one query tile at a time, tile A then tile B for every key
// tile. Warps w and w + 4 share TMEM lane quarter w % 4 (query rows 32 (w % 4) ... + 31); warp
// w takes key columns 0..63 of the key tile and warp w + 4 columns 64..127. So the softmax of
// one tile has two warps on every sub-partition while the MMAs of the other tile run, instead
// of two tiles' softmaxes sharing the sub-partitions at once.
struct TileState {
  float m_run;       // running max of scaled scores (log2 units), kept key tiles only
  float m_use;       // exponent reference of l and O (trails m_run by <= 8)
  float l;           // this thread's half of the row sum, relative to m_use
  int pv_count;      // kept key tiles so far
  uint32_t skipped;  // skipped key tiles so far (counted by the leader thread)
};

__device__ __forceinline__ void swap_state(TileState& a, TileState& b) {
  const TileState tmp = a;
  a = b;
  b = tmp;
}

template <bool kVarlen, bool kMaxProb>
__device__ __forceinline__ void run_softmax(Smem& sm, uint32_t tmem, const FwdParams& p, const Geo& g,
                                            int b, int h, int qt0) {
  const Lens<kVarlen> L{p, g};
  volatile uint32_t* abort = &sm.abort;
  const int warp = threadIdx.x >> 5;
  const int wq = warp & 3;                // TMEM lane quarter
  const int half = warp >> 2;             // key columns 64 * half ... + 63; O features likewise
  const int lane = threadIdx.x & 31;
  const int row = wq * 32 + lane;         // query row inside the tile == TMEM lane
  const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
  const bool leader = threadIdx.x == 0;
  TileState cur{-INFINITY, -INFINITY, 0.f, 0, 0u};  // the tile of the current step
  TileState oth = cur;                              // the other tile
  bool failed = false;
  bool left_early = false;

  for (int step = 0; step < 2 * L.nK(); ++step) {
    const int t = step & 1;
    const int j = step >> 1;
    const int qt = qt0 + t;
    const bool row_valid = qt * kTile + row < g.Sq;
    const uint32_t t_s = tmem + lane_base + col_s(t);
    bool pass = true;
    float hmax = -INFINITY;
    uint32_t sr[64];
    if (!failed) {
      const bool ok = wait_bar(smem_u32(&sm.s_full[t]), j & 1, abort, kErrSoftmax);
      failed = !__all_sync(0xffffffffu, ok);
    }
    if (!failed) {
      tc_fence_after();
      tmem_ld64(t_s + half * 64, sr);
      const int valid_keys = L.Sk() - j * kTile - half * 64;
      if (valid_keys < 64) {
#pragma unroll
        for (int c = 0; c < 64; ++c)
          if (c >= valid_keys) sr[c] = __float_as_uint(-INFINITY);
      }
      float mx0 = -INFINITY, mx1 = -INFINITY, mx2 = -INFINITY, mx3 = -INFINITY;
#pragma unroll
      for (int c = 0; c < 64; c += 8) {
        mx0 = fmax3(mx0, __uint_as_float(sr[c + 0]), __uint_as_float(sr[c + 1]));
        mx1 = fmax3(mx1, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
        mx2 = fmax3(mx2, __uint_as_float(sr[c + 4]), __uint_as_float(sr[c + 5]));
        mx3 = fmax3(mx3, __uint_as_float(sr[c + 6]), __uint_as_float(sr[c + 7]));
      }
      hmax = fmax3(mx0, mx1, fmaxf(mx2, mx3));
      sm.hmax[t][half][row] = hmax;
      // A row passes when both of its halves pass; rows past Sq do not exist and always pass.
      pass = !row_valid || (hmax * p.scale_log2 - cur.m_run < L.log2_lambda());
    } else {
      sm.quit[t][j & 1] = 1u;
    }
    // The skip test over all 128 rows (both halves of each); the barrier also publishes hmax.
    const bool skip = bar_and<2 * kSoftmaxThreads>(1u + static_cast<uint32_t>(t), pass);
    if (*reinterpret_cast<volatile uint32_t*>(&sm.quit[t][j & 1])) {  // written only before this barrier
      left_early = true;
      break;
    }
    do {
      if (leader) {
        // Publish the decision: the producer loads V_j only if some tile keeps key tile j,
        // and the MMA issues P V only for a kept tile.
        sm.skip_flag[t][j & 1] = skip ? 1u : 0u;
        mbar_arrive(smem_u32(&sm.dec[t][j & 1]));
        if (qt < g.nQ && p.skip_mask)
          p.skip_mask[((static_cast<size_t>(b) * p.H + h) * p.nQ + qt) * static_cast<size_t>(p.nK) + j] = skip ? 1 : 0;
      }
      if (skip) {
        if (leader) ++cur.skipped;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm.p_ready[t]));
        break;
      }

      // Kept key tile: online-softmax update with the full row max.
      const float tm2 = fmaxf(hmax, sm.hmax[t][half ^ 1][row]) * p.scale_log2;
      const float m_new = fmaxf(cur.m_run, tm2);
      cur.m_run = m_new;
      float alpha = 1.f;
      if (m_new - cur.m_use > kRescaleThreshold) {
        alpha = ex2_approx(cur.m_use - m_new);  // 0 for the first kept tile
        cur.m_use = m_new;
      }
      // P = exp2(s * scale * log2 e - m_use) for this thread's 64 keys, two per packed f32x2
      // FMA; P (bf16, keys 2c and 2c + 1 in column c) overwrites columns 32 half ... + 31 of
      // S_j. (Every thread read its scores before the vote barrier.)
      const uint64_t scale2 = pack_f32x2(p.scale_log2, p.scale_log2);
      const uint64_t nref2 = pack_f32x2(-cur.m_use, -cur.m_use);
      uint64_t sum_a = pack_f32x2(0.f, 0.f), sum_b = sum_a;
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const uint64_t x2 =
            fma_f32x2(pack_f32x2(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), scale2, nref2);
        float x0, x1;
        unpack_f32x2(x2, x0, x1);
        const float p0 = ex2_approx(x0);
        const float p1 = ex2_approx(x1);
        if (c & 1)
          sum_b = add_f32x2(sum_b, pack_f32x2(p0, p1));
        else
          sum_a = add_f32x2(sum_a, pack_f32x2(p0, p1));
        pk[c] = pack_bf16(p0, p1);
      }
      tmem_st32(t_s + half * 32, pk);
      tmem_st_wait();
      {
        float a0, a1, b0, b1;
        unpack_f32x2(sum_a, a0, a1);
        unpack_f32x2(sum_b, b0, b1);
        cur.l = cur.l * alpha + ((a0 + a1) + (b0 + b1));
      }
      // O (this thread's 64 features) is rescaled only by warps that need it. Every earlier
      // P V of this tile has completed: S_j, which this thread waited for, was committed
      // after them.
      if (cur.pv_count > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        const uint32_t t_o = tmem + lane_base + col_o(t) + half * 64;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t r[32];
          tmem_ld32(t_o + c * 32, r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st32(t_o + c * 32, r);
        }
        tmem_st_wait();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.p_ready[t]));
      ++cur.pv_count;
    } while (false);
    swap_state(cur, oth);
  }
  if (left_early) return;

  // Epilogue: after 2 nK steps `cur` holds tile A and `oth` tile B. The two halves of each
  // row combine their sums (same exponent reference), then write their 64 features of O.
  sm.lpart[0][half][row] = cur.l;
  sm.lpart[1][half][row] = oth.l;
  bar_sync_n<2 * kSoftmaxThreads>(3u);
  const bool ok = failed ? false : wait_bar(smem_u32(&sm.o_done[0]), 0, abort, kErrSoftmax) &&
                                       wait_bar(smem_u32(&sm.o_done[1]), 0, abort, kErrSoftmax);
  if (!__all_sync(0xffffffffu, ok)) return;
  tc_fence_after();
#pragma unroll 1
  for (int t = 0; t < kQTiles; ++t) {
    const TileState st = t ? oth : cur;
    const int qt = qt0 + t;
    const int q_row = qt * kTile + row;
    const bool tile_exists = qt < g.nQ;
    const bool row_valid = q_row < g.Sq;
    if (leader && tile_exists && p.skip_counts && st.skipped)
      atomicAdd(&p.skip_counts[static_cast<size_t>(b) * p.H + h], st.skipped);
    if (!tile_exists || st.pv_count == 0) continue;
    const float l = st.l + sm.lpart[t][half ^ 1][row];
    const float inv_l = 1.f / l;
    const uint32_t t_o = tmem + lane_base + col_o(t) + half * 64;
    __nv_bfloat16* orow =
        p.o + ((out_tok0<kVarlen>(p, g, b) + (row_valid ? q_row : 0)) * p.H + h) * kHeadDim + half * 64;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      uint32_t r[32];
      tmem_ld32(t_o + c * 32, r);
      if (row_valid) {
        uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint4 w;
          w.x = pack_bf16(__uint_as_float(r[8 * i + 0]) * inv_l, __uint_as_float(r[8 * i + 1]) * inv_l);
          w.y = pack_bf16(__uint_as_float(r[8 * i + 2]) * inv_l, __uint_as_float(r[8 * i + 3]) * inv_l);
          w.z = pack_bf16(__uint_as_float(r[8 * i + 4]) * inv_l, __uint_as_float(r[8 * i + 5]) * inv_l);
          w.w = pack_bf16(__uint_as_float(r[8 * i + 6]) * inv_l, __uint_as_float(r[8 * i + 7]) * inv_l);
          dst[i] = w;
        }
      }
    }
    if (half == 0 && row_valid) {
      const size_t stat0 = stat_base<kVarlen>(p, g, b, h);
      if (p.lse) p.lse[stat0 + q_row] = (st.m_use + log2f(l)) * kLn2;
      // The largest softmax weight of the row, exp(m - m) / l with l relative to the row
      // max m ("video-attention", "max_prob = 1 / l_i"): 2^(m_run - m_use) / l here.
      if (kMaxProb) p.max_prob[stat0 + q_row] = ex2_approx(st.m_run - st.m_use) * inv_l;
    }
  }
}

// One instance per feature set (packed documents, max_prob output, e4m3 scores), so that the
// plain fixed-length instance keeps the code generation of a kernel without them.
template <bool kVarlen, bool kMaxProb, bool kFp8>
__global__ void __launch_bounds__(kThreads, 1)
    blasst_fwd_sm103a(const __grid_constant__ CUtensorMap tmap_q,
                      const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // Blocks start in blockIdx.x order: the last query tiles, which keep the longest prefix of key
  // tiles when the test skips, go first, so the short ones fill the last wave.
  const int qt0 = (gridDim.x - 1 - blockIdx.x) * kQTiles, h = blockIdx.y, b = blockIdx.z;
  const Geo g = make_geo<kVarlen>(p, b, h);
  if (qt0 * kTile >= g.Sq) return;  // a packed document shorter than this CTA's first row
  if (g.Sk == 0) {
    // A document without keys: no softmax is defined; write O = 0, lse = -inf, max_prob = 0.
    if (warp < kQTiles * kSoftmaxWarps) {
      const int q_row = (qt0 + warp / kSoftmaxWarps) * kTile + (threadIdx.x & (kSoftmaxThreads - 1));
      if (q_row < g.Sq) {
        uint4* dst = reinterpret_cast<uint4*>(p.o + ((out_tok0<kVarlen>(p, g, b) + q_row) * p.H + h) * kHeadDim);
        for (int i = 0; i < kHeadDim / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
        if (p.lse) p.lse[stat_base<kVarlen>(p, g, b, h) + q_row] = -INFINITY;
        if (p.max_prob) p.max_prob[stat_base<kVarlen>(p, g, b, h) + q_row] = 0.f;
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm.q_full), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.k_full[s]), 1);
      mbar_init(smem_u32(&sm.v_full[s]), 1);
    }
    for (int t = 0; t < kQTiles; ++t) {
      mbar_init(smem_u32(&sm.s_full[t]), 1);
      mbar_init(smem_u32(&sm.dec[t][0]), 1);
      mbar_init(smem_u32(&sm.dec[t][1]), 1);
      mbar_init(smem_u32(&sm.p_ready[t]), kQTiles * kSoftmaxWarps);
      mbar_init(smem_u32(&sm.o_done[t]), 1);
      sm.skip_flag[t][0] = 0u;
      sm.skip_flag[t][1] = 0u;
      sm.quit[t][0] = 0u;
      sm.quit[t][1] = 0u;
    }
    mbar_init(smem_u32(&sm.drain), 1);
    sm.abort = 0u;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&sm.tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // Nothing computed above stays live past the role branch: values that cross it would have
  // to survive the softmax region at its register limit, and the compiler would spill them
  // and reload them inside the MMA issue loop. The join below re-derives what it needs.
  if (warp >= kMmaWarp) {
    regs_decrease<kControlRegs>();
    if (warp == kLoadWarp) {
      if (lane == 0) run_producer<kVarlen, kFp8>(sm, &tmap_q, &tmap_k, &tmap_v, p, g, h, qt0);
      __syncwarp();
    } else if (warp == kMmaWarp) {
      run_mma<kVarlen, kFp8>(sm, sm.tmem_base, p, g);
    }
  } else {
    regs_increase<kSoftmaxRegs>();
    run_softmax<kVarlen, kMaxProb>(sm, sm.tmem_base, p, g, b, h, qt0);
  }

  tc_fence_before();
  __syncthreads();
  // A wait that gave up left its role's bit in the abort word: report it device-wide and to the
  // caller's status word.
  if (threadIdx.x == 0) {
    const uint32_t bits = *reinterpret_cast<volatile uint32_t*>(&sm.abort);
    if (bits) report_error(p.status, bits);
  }
  if ((threadIdx.x >> 5) == kMmaWarp) {
    Smem& sm2 = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                         ~static_cast<uintptr_t>(1023));
    tc_fence_after();
    tmem_dealloc(*reinterpret_cast<volatile uint32_t*>(&sm2.tmem_base), kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// [B, S, H, 128] viewed as a 4-D tensor (d, H, S, B); boxes of 128 bytes of features (64 bf16
// or 128 e4m3) x 1 head x 128 tokens x 1 batch, 128-byte swizzled. Tokens past S read as zero.
bool encode_bshd(CUtensorMap* map, const void* base, int B, int S, int H, bool e4m3 = false) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
  const cuuint64_t row = static_cast<cuuint64_t>(kHeadDim) * (e4m3 ? 1 : 2);
  const cuuint64_t strides[3] = {row, row * static_cast<cuuint64_t>(H),
                                 row * static_cast<cuuint64_t>(H) * static_cast<cuuint64_t>(S)};
  const cuuint32_t box[4] = {e4m3 ? 128u : 64u, 1, static_cast<cuuint32_t>(kTile), 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  return fn(map, e4m3 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
            const_cast<void*>(base), dims, strides, box,
            estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor descriptors are a pure function of (address, shape, format), so a small per-process
// table keeps the last ones encoded and repeated calls on the same tensors encode nothing.
struct TmapKey {
  const void* base;
  int B, S, H;
  bool e4m3;
  bool operator==(const TmapKey& o) const {
    return base == o.base && B == o.B && S == o.S && H == o.H && e4m3 == o.e4m3;
  }
};
constexpr int kTmapCacheSize = 48;
struct TmapCache {
  std::mutex mutex;
  TmapKey key[kTmapCacheSize] = {};
  CUtensorMap map[kTmapCacheSize];
  bool used[kTmapCacheSize] = {};
  int next = 0;
};
TmapCache g_tmaps;
std::atomic<uint64_t> g_tmap_encodes{0};

bool cached_bshd(CUtensorMap* map, const void* base, int B, int S, int H, bool e4m3) {
  const TmapKey key{base, B, S, H, e4m3};
  std::lock_guard<std::mutex> lock(g_tmaps.mutex);
  for (int i = 0; i < kTmapCacheSize; ++i) {
    if (g_tmaps.used[i] && g_tmaps.key[i] == key) {
      *map = g_tmaps.map[i];
      return true;
    }
  }
  if (!encode_bshd(map, base, B, S, H, e4m3)) return false;
  g_tmap_encodes.fetch_add(1, std::memory_order_relaxed);
  const int slot = g_tmaps.next;
  g_tmaps.next = (slot + 1) % kTmapCacheSize;
  g_tmaps.key[slot] = key;
  g_tmaps.map[slot] = *map;
  g_tmaps.used[slot] = true;
  return true;
}

// The key tile whose copy the producer withholds (test of the bounded waits; -1: off).
std::atomic<int> g_withhold_k{-1};

// The instance for feature bits (1 = packed documents, 2 = max_prob, 4 = e4m3 Q / K).
// lambda = 0 runs the same instances: no tile passes the test and every one is kept.
template <int kBits>
const void* instance() {
  return reinterpret_cast<const void*>(
      blasst_fwd_sm103a<(kBits & 1) != 0, (kBits & 2) != 0, (kBits & 4) != 0>);
}
constexpr int kInstances = 8;
const void* kernel_for(int bits) {
  switch (bits & 7) {
    case 0: return instance<0>();
    case 1: return instance<1>();
    case 2: return instance<2>();
    case 3: return instance<3>();
    case 4: return instance<4>();
    case 5: return instance<5>();
    case 6: return instance<6>();
    default: return instance<7>();
  }
}

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
int g_dev_state[kMaxDevices];  // 0 unknown, 1 ready, 2 unsupported

blasst_status prepare_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return BLASST_ERR_UNSUPPORTED_DEVICE;
  }
  if (dev >= kMaxDevices) return BLASST_ERR_UNSUPPORTED_DEVICE;
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  if (g_dev_state[dev] == 1) return BLASST_OK;
  if (g_dev_state[dev] == 2) return BLASST_ERR_UNSUPPORTED_DEVICE;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
    cudaGetLastError();
    return BLASST_ERR_UNSUPPORTED_DEVICE;
  }
  if (major != 10 || minor != 3) {
    g_dev_state[dev] = 2;
    return BLASST_ERR_UNSUPPORTED_DEVICE;
  }
  bool attr_ok = true;
  for (int i = 0; i < kInstances; ++i)
    attr_ok = attr_ok && cudaFuncSetAttribute(kernel_for(i), cudaFuncAttributeMaxDynamicSharedMemorySize,
                                              static_cast<int>(kSmemBytes)) == cudaSuccess;
  if (!attr_ok) {
    cudaGetLastError();
    return BLASST_ERR_LAUNCH;
  }
  g_dev_state[dev] = 1;
  return BLASST_OK;
}

bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; }

}  // namespace
}  // namespace blasst

namespace blasst {
namespace {

blasst_status launch(const blasst_fwd_args& a) {
  const bool varlen = a.cu_seqlens_q != nullptr || a.cu_seqlens_k != nullptr;
  // ---- argument checks: no CUDA call happens before all of them pass
  if (!a.q || !a.k || !a.v || !a.o) return BLASST_ERR_INVALID_ARG;
  if (a.B <= 0 || a.H <= 0 || a.Sq <= 0 || a.Sk <= 0 || a.B > 65535 || a.H > 65535) return BLASST_ERR_INVALID_ARG;
  if (a.d != kHeadDim) return BLASST_ERR_INVALID_ARG;
  if (!std::isfinite(a.scale) || !(a.scale > 0.f)) return BLASST_ERR_INVALID_ARG;
  if (!std::isfinite(a.factor) || !(a.factor >= 0.f)) return BLASST_ERR_INVALID_ARG;
  if (a.qk_format != BLASST_QK_BF16 && a.qk_format != BLASST_QK_E4M3) return BLASST_ERR_INVALID_ARG;
  const bool e4m3 = a.qk_format == BLASST_QK_E4M3;
  double qk_descale = 1.0;
  if (e4m3) {
    if (!std::isfinite(a.q_descale) || !(a.q_descale > 0.f) || !std::isfinite(a.k_descale) ||
        !(a.k_descale > 0.f))
      return BLASST_ERR_INVALID_ARG;
    qk_descale = static_cast<double>(a.q_descale) * static_cast<double>(a.k_descale);
  }
  if (!aligned(a.q, 16) || !aligned(a.k, 16) || !aligned(a.v, 16) || !aligned(a.o, 16))
    return BLASST_ERR_INVALID_ARG;
  if ((a.lse && !aligned(a.lse, 4)) || (a.max_prob && !aligned(a.max_prob, 4))) return BLASST_ERR_INVALID_ARG;
  if (a.status && !aligned(a.status, 4)) return BLASST_ERR_INVALID_ARG;
  if (a.min_seq_len < 0) return BLASST_ERR_INVALID_ARG;
  if (varlen) {
    if (!a.cu_seqlens_q || !a.cu_seqlens_k || !aligned(a.cu_seqlens_q, 4) || !aligned(a.cu_seqlens_k, 4))
      return BLASST_ERR_INVALID_ARG;
    if (a.skip_mask_dbg) return BLASST_ERR_INVALID_ARG;  // the mask layout needs one length
    if (a.max_seqlen_q <= 0 || a.max_seqlen_k <= 0 || a.max_seqlen_q > a.Sq || a.max_seqlen_k > a.Sk)
      return BLASST_ERR_INVALID_ARG;
  }
  // byte strides of the 4-D views must stay below 2^40 (TMA limit)
  const double batch_stride = 256.0 * a.H * static_cast<double>(a.Sq > a.Sk ? a.Sq : a.Sk);
  if (batch_stride >= 1099511627776.0) return BLASST_ERR_INVALID_ARG;

  const blasst_status ds = prepare_device();
  if (ds != BLASST_OK) return ds;

  // Fixed length: [B, S, H, 128] views. Packed documents: one [1, T, H, 128] view of all tokens.
  const int tb = varlen ? 1 : a.B;
  CUtensorMap tq, tk, tv;
  if (!cached_bshd(&tq, a.q, tb, a.Sq, a.H, e4m3) || !cached_bshd(&tk, a.k, tb, a.Sk, a.H, e4m3) ||
      !cached_bshd(&tv, a.v, tb, a.Sk, a.H, false))
    return BLASST_ERR_LAUNCH;

  FwdParams p{};
  p.B = a.B;
  p.H = a.H;
  p.Sq = varlen ? a.max_seqlen_q : a.Sq;  // longest entry: sizes the grid
  p.Sk = varlen ? a.max_seqlen_k : a.Sk;  // the KV length lambda is normalised by
  p.nQ = (p.Sq + kTile - 1) / kTile;      // query tiles; CTAs hold kQTiles each
  p.nK = (p.Sk + kTile - 1) / kTile;
  p.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * qk_descale * 1.4426950408889634);
  p.log2_lambda = a.factor > 0.f ? static_cast<float>(std::log2(static_cast<double>(a.factor) / p.Sk))
                                 : -INFINITY;
  if (!varlen && a.Sk < a.min_seq_len) p.log2_lambda = -INFINITY;  // one length: decided here
  p.o = static_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.max_prob = a.max_prob;
  p.skip_counts = a.skip_counts;
  p.skip_mask = a.skip_mask_dbg;
  p.cu_q = varlen ? a.cu_seqlens_q : nullptr;
  p.cu_k = varlen ? a.cu_seqlens_k : nullptr;
  p.Tq = a.Sq;
  p.Tk = a.Sk;
  p.min_seq_len = a.min_seq_len;
  // Test of the bounded device waits (blasst_debug_withhold_key_tile): the producer skips the
  // copy of this key tile, so the waits on it give up after their time limit.
  p.withhold_k = g_withhold_k.load(std::memory_order_relaxed);
  p.status = a.status;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(a.stream);
  if (a.skip_counts &&
      cudaMemsetAsync(a.skip_counts, 0, sizeof(uint32_t) * static_cast<size_t>(a.B) * a.H, st) != cudaSuccess) {
    cudaGetLastError();
    return BLASST_ERR_LAUNCH;
  }
  if (a.status && cudaMemsetAsync(a.status, 0, sizeof(uint32_t), st) != cudaSuccess) {
    cudaGetLastError();
    return BLASST_ERR_LAUNCH;
  }
  void* args[] = {&tq, &tk, &tv, &p};
  const void* kernel = kernel_for((varlen ? 1 : 0) | (a.max_prob ? 2 : 0) | (e4m3 ? 4 : 0));
  const cudaError_t e = cudaLaunchKernel(kernel,
                                         dim3((p.nQ + kQTiles - 1) / kQTiles, a.H, a.B), dim3(kThreads), args,
                                         kSmemBytes, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return BLASST_ERR_LAUNCH;
  }
  return BLASST_OK;
}

}  // namespace
}  // namespace blasst

namespace blasst {
namespace {

// ------------------------------------------------------------------ host-buffer streaming
constexpr size_t kWsAlign = 256;
size_t round_up(size_t x) { return (x + kWsAlign - 1) / kWsAlign * kWsAlign; }

// One workspace slot holds a head group's q, k, v, o and lse.
struct HostSlot {
  size_t q, k, v, o, lse, bytes;  // byte offsets inside the slot, and its size
};
HostSlot host_slot(int B, int Sq, int Sk, int hg) {
  HostSlot s{};
  const size_t row = static_cast<size_t>(hg) * kHeadDim * 2;
  s.q = 0;
  s.o = s.q + round_up(static_cast<size_t>(B) * Sq * row);
  s.k = s.o + round_up(static_cast<size_t>(B) * Sq * row);
  s.v = s.k + round_up(static_cast<size_t>(B) * Sk * row);
  s.lse = s.v + round_up(static_cast<size_t>(B) * Sk * row);
  s.bytes = s.lse + round_up(static_cast<size_t>(B) * hg * Sq * sizeof(float));
  return s;
}

bool host_dims_ok(int B, int H, int Sq, int Sk, int hg) {
  return B > 0 && H > 0 && Sq > 0 && Sk > 0 && B <= 65535 && H <= 65535 && hg >= 1 && hg <= H;
}

// Streams and events of the host-buffer call, one set per device, made at its first use there.
struct HostPipe {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr, comp[2] = {};
  cudaEvent_t start = nullptr, in_done[2] = {}, comp_done[2] = {}, out_done[2] = {};
};
HostPipe g_pipe[kMaxDevices];
std::mutex g_pipe_mutex;

bool make_pipe(HostPipe& hp) {
  if (hp.ready) return true;
  bool ok = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&hp.comp[0], cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&hp.comp[1], cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming) == cudaSuccess;
  for (int i = 0; i < 2 && ok; ++i)
    ok = cudaEventCreateWithFlags(&hp.in_done[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&hp.comp_done[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&hp.out_done[i], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    return false;
  }
  hp.ready = true;
  return true;
}

blasst_status launch_host(const blasst_host_args& a) {
  // ---- argument checks: no CUDA call happens before all of them pass
  if (!a.q || !a.k || !a.v || !a.o || !a.workspace) return BLASST_ERR_INVALID_ARG;
  if (!host_dims_ok(a.B, a.H, a.Sq, a.Sk, a.heads_per_group) || a.d != kHeadDim) return BLASST_ERR_INVALID_ARG;
  if (!std::isfinite(a.scale) || !(a.scale > 0.f)) return BLASST_ERR_INVALID_ARG;
  if (!std::isfinite(a.factor) || !(a.factor >= 0.f)) return BLASST_ERR_INVALID_ARG;
  if (!aligned(a.workspace, kWsAlign)) return BLASST_ERR_INVALID_ARG;
  const int hg = a.heads_per_group;
  const HostSlot slot = host_slot(a.B, a.Sq, a.Sk, hg);
  if (a.workspace_bytes < 2 * slot.bytes) return BLASST_ERR_INVALID_ARG;
  const double batch_stride = 256.0 * a.H * static_cast<double>(a.Sq > a.Sk ? a.Sq : a.Sk);
  if (batch_stride >= 1099511627776.0) return BLASST_ERR_INVALID_ARG;

  const blasst_status ds = prepare_device();
  if (ds != BLASST_OK) return ds;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return BLASST_ERR_LAUNCH;
  }
  std::lock_guard<std::mutex> lock(g_pipe_mutex);
  HostPipe& hp = g_pipe[dev];
  if (!make_pipe(hp)) return BLASST_ERR_LAUNCH;

  cudaStream_t cs = reinterpret_cast<cudaStream_t>(a.stream);
  const size_t hrow = static_cast<size_t>(a.H) * kHeadDim * 2;  // host bytes per (batch, token)
  bool ok = cudaEventRecord(hp.start, cs) == cudaSuccess &&
            cudaStreamWaitEvent(hp.in, hp.start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(hp.out, hp.start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(hp.comp[0], hp.start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(hp.comp[1], hp.start, 0) == cudaSuccess;
  // Groups of heads: sizes 1, 2, 3, 5, 8, ... (about 1.5 times the previous) up to hg, so that
  // each group's copy-in takes no longer than the previous group's kernel (a short pipeline
  // fill), and a single head last (a short drain). The two workspace slots have a compute
  // stream each, so the kernel of one group can start on the SMs that the previous group's
  // kernel is leaving (no tail between launches).
  blasst_status kst = BLASST_OK;
  int want = 1;
  for (int g = 0, h0 = 0, hc = 0; h0 < a.H && ok;
       ++g, h0 += hc, want = want + (want + 1) / 2 < hg ? want + (want + 1) / 2 : hg) {
    const int rem = a.H - h0;
    hc = rem > want ? want : (rem > 1 && g > 0 ? rem - 1 : rem);
    const int s = g & 1;
    const size_t crow = static_cast<size_t>(hc) * kHeadDim * 2;  // device bytes per (batch, token)
    uint8_t* base = static_cast<uint8_t*>(a.workspace) + s * slot.bytes;
    const size_t hoff = static_cast<size_t>(h0) * kHeadDim * 2;
    // The kernel of group g - 2 read this slot's q, k, v; the copy-out of group g - 2 read its o, lse.
    if (g >= 2) ok = cudaStreamWaitEvent(hp.in, hp.comp_done[s], 0) == cudaSuccess;
    ok = ok &&
         cudaMemcpy2DAsync(base + slot.q, crow, static_cast<const uint8_t*>(a.q) + hoff, hrow, crow,
                           static_cast<size_t>(a.B) * a.Sq, cudaMemcpyHostToDevice, hp.in) == cudaSuccess &&
         cudaMemcpy2DAsync(base + slot.k, crow, static_cast<const uint8_t*>(a.k) + hoff, hrow, crow,
                           static_cast<size_t>(a.B) * a.Sk, cudaMemcpyHostToDevice, hp.in) == cudaSuccess &&
         cudaMemcpy2DAsync(base + slot.v, crow, static_cast<const uint8_t*>(a.v) + hoff, hrow, crow,
                           static_cast<size_t>(a.B) * a.Sk, cudaMemcpyHostToDevice, hp.in) == cudaSuccess &&
         cudaEventRecord(hp.in_done[s], hp.in) == cudaSuccess &&
         cudaStreamWaitEvent(hp.comp[s], hp.in_done[s], 0) == cudaSuccess;
    // The copy-out of group g - 2 read this slot's o and lse.
    if (ok && g >= 2) ok = cudaStreamWaitEvent(hp.comp[s], hp.out_done[s], 0) == cudaSuccess;
    if (!ok) break;
    blasst_fwd_args fa{};
    fa.struct_size = sizeof(fa);
    fa.q = base + slot.q;
    fa.k = base + slot.k;
    fa.v = base + slot.v;
    fa.o = base + slot.o;
    fa.lse = a.lse ? reinterpret_cast<float*>(base + slot.lse) : nullptr;
    fa.B = a.B;
    fa.H = hc;
    fa.Sq = a.Sq;
    fa.Sk = a.Sk;
    fa.d = a.d;
    fa.scale = a.scale;
    fa.factor = a.factor;
    fa.stream = reinterpret_cast<struct CUstream_st*>(hp.comp[s]);
    kst = launch(fa);
    if (kst != BLASST_OK) break;
    ok = cudaEventRecord(hp.comp_done[s], hp.comp[s]) == cudaSuccess &&
         cudaStreamWaitEvent(hp.out, hp.comp_done[s], 0) == cudaSuccess &&
         cudaMemcpy2DAsync(static_cast<uint8_t*>(a.o) + hoff, hrow, base + slot.o, crow, crow,
                           static_cast<size_t>(a.B) * a.Sq, cudaMemcpyDeviceToHost, hp.out) == cudaSuccess;
    if (ok && a.lse)  // device [B, hc, Sq] -> host rows (b H + h0) Sq ... of [B, H, Sq]
      ok = cudaMemcpy2DAsync(a.lse + static_cast<size_t>(h0) * a.Sq, static_cast<size_t>(a.H) * a.Sq * sizeof(float),
                             base + slot.lse, static_cast<size_t>(hc) * a.Sq * sizeof(float),
                             static_cast<size_t>(hc) * a.Sq * sizeof(float), a.B, cudaMemcpyDeviceToHost,
                             hp.out) == cudaSuccess;
    ok = ok && cudaEventRecord(hp.out_done[s], hp.out) == cudaSuccess;
  }
  // Later work on the caller's stream starts after the last copy back.
  const bool tail = cudaEventRecord(hp.out_done[0], hp.out) == cudaSuccess &&
                    cudaStreamWaitEvent(cs, hp.out_done[0], 0) == cudaSuccess;
  if (kst != BLASST_OK) return kst;
  if (!ok || !tail) {
    cudaGetLastError();
    return BLASST_ERR_LAUNCH;
  }
  return BLASST_OK;
}

}  // namespace

blasst_status run_host_pipeline(const blasst_host_args& a) { return launch_host(a); }

blasst_status check_device() { return prepare_device(); }

}  // namespace blasst

extern "C" size_t blasst_host_workspace_bytes(int B, int H, int Sq, int Sk, int heads_per_group) {
  if (!blasst::host_dims_ok(B, H, Sq, Sk, heads_per_group)) return 0;
  return 2 * blasst::host_slot(B, Sq, Sk, heads_per_group).bytes;
}

extern "C" blasst_status blasst_attn_fwd_host(const blasst_host_args* args) {
  if (!args || args->struct_size != sizeof(blasst_host_args)) return BLASST_ERR_INVALID_ARG;
  return blasst::launch_host(*args);
}

extern "C" blasst_status blasst_attn_fwd(const void* q, const void* k, const void* v, void* o,
                                         float* lse, int B, int H, int Sq, int Sk, int d,
                                         float scale, float factor, struct CUstream_st* stream,
                                         uint32_t* skip_counts, uint8_t* skip_mask_dbg) {
  blasst_fwd_args a{};
  a.struct_size = sizeof(a);
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.H = H;
  a.Sq = Sq;
  a.Sk = Sk;
  a.d = d;
  a.scale = scale;
  a.factor = factor;
  a.stream = stream;
  a.skip_counts = skip_counts;
  a.skip_mask_dbg = skip_mask_dbg;
  return blasst::launch(a);
}

extern "C" blasst_status blasst_attn_fwd_ex(const blasst_fwd_args* args) {
  if (!args) return BLASST_ERR_INVALID_ARG;
  if (args->struct_size == offsetof(blasst_fwd_args, status)) {
    // the layout before the status word: copy what the caller has, status NULL
    blasst_fwd_args a{};
    std::memcpy(&a, args, offsetof(blasst_fwd_args, status));
    a.status = nullptr;
    return blasst::launch(a);
  }
  if (args->struct_size != sizeof(blasst_fwd_args)) return BLASST_ERR_INVALID_ARG;
  return blasst::launch(*args);
}

extern "C" const char* blasst_status_string(blasst_status s) {
  switch (s) {
    case BLASST_OK: return "ok";
    case BLASST_ERR_INVALID_ARG: return "invalid argument";
    case BLASST_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
    case BLASST_ERR_LAUNCH: return "CUDA launch or set-up failure";
    case BLASST_ERR_TIMEOUT: return "a device-side wait timed out or packed-document offsets were invalid";
    case BLASST_ERR_TOO_LARGE: return "the problem does not fit the library's fixed-size buffer";
  }
  return "unknown status";
}

extern "C" blasst_status blasst_device_error(uint32_t* word, int clear) {
  if (!word) return BLASST_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return BLASST_ERR_LAUNCH;
  }
  uint32_t w = 0;
  if (cudaMemcpyFromSymbol(&w, blasst::g_error_word, sizeof w) != cudaSuccess) {
    cudaGetLastError();
    return BLASST_ERR_LAUNCH;
  }
  if (clear) {
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(blasst::g_error_word, &zero, sizeof zero) != cudaSuccess) {
      cudaGetLastError();
      return BLASST_ERR_LAUNCH;
    }
  }
  *word = w;
  return w ? BLASST_ERR_TIMEOUT : BLASST_OK;
}

extern "C" int blasst_version(void) { return 10300; }

extern "C" blasst_status blasst_debug_withhold_key_tile(int tile) {
  if (tile < -1) return BLASST_ERR_INVALID_ARG;
  blasst::g_withhold_k.store(tile, std::memory_order_relaxed);
  return BLASST_OK;
}

extern "C" uint64_t blasst_tensor_map_encodes(void) {
  return blasst::g_tmap_encodes.load(std::memory_order_relaxed);
}
