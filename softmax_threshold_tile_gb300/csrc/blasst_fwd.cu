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
// One CTA owns one 128-row query tile of one (batch, head) and streams all key
// tiles through a warp-specialised pipeline:
//   warps 0-3  softmax: one query row per thread (= TMEM lane). tcgen05.ld of
//              S_j, row max, CTA-subset AND-vote on the skip test, exp2 of the
//              kept tile written back into TMEM as bf16 P (aliasing S_j),
//              conditional O rescale, epilogue (O / l -> bf16, lse).
//   warp 4     MMA: one thread issues tcgen05.mma. S_{j+1} = Q K_{j+1}^T is
//              issued before waiting for tile j's decision, so the tensor pipe
//              computes the next scores while the softmax warps vote; then
//              O += P_j V_j (A operand from TMEM) only for kept tiles.
//   warp 5     TMA producer: Q once, K/V tiles through a 2-stage ring.
// TMEM (512 columns): S0 [0,128), S1 [128,256), O [256,384).
// Shared memory: Q 32 KiB, K 2 x 32 KiB, V 2 x 32 KiB, all 128-byte swizzled.
//
// Numerics: scores are fp32 from bf16 operands; the test is evaluated in log2
// units, (tile_max - running_max) * scale * log2(e) < log2(lambda), which is the
// pages' log-space test scaled by log2(e). P is rounded to bf16 for P V; l and O
// accumulate in fp32. The exponent reference m_use trails the true running max
// by at most 8 (log2 units), so O is rescaled only when the max grows by more
// than that; the skip test always uses the true running max.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "blasst.h"
#include "sm103_ptx.cuh"

namespace blasst {
namespace {

using namespace ptx;

constexpr int kTile = 128;      // query rows per query tile == keys per key tile
constexpr int kHeadDim = 128;   // d
constexpr int kSoftmaxWarps = 4;
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;
constexpr int kMmaWarp = 4;
constexpr int kLoadWarp = 5;
constexpr int kThreads = 192;
constexpr int kStages = 2;
constexpr uint32_t kTileBytes = kTile * kHeadDim * 2;  // one bf16 128 x 128 tile
constexpr uint32_t kHalfBytes = kTileBytes / 2;        // 128 rows x 64 features (128-B rows)
constexpr uint32_t kTmemCols = 512;
__host__ __device__ constexpr uint32_t col_s(int buf) { return static_cast<uint32_t>(buf) * 128u; }  // S0, S1
constexpr uint32_t kColO = 256;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2 = 0.693147180559945309f;
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // a single wait may last at most 2 s
constexpr uint64_t kDrainTimeoutNs = 50000000ull;   // waits for in-flight copies / MMAs at exit

// Bits of the device error word: which role gave up waiting.
constexpr uint32_t kErrProducer = 1u << 0;
constexpr uint32_t kErrMma = 1u << 1;
constexpr uint32_t kErrSoftmax = 1u << 2;
constexpr uint32_t kErrDrain = 1u << 3;

__device__ uint32_t g_error_word;

struct alignas(1024) Smem {
  uint8_t q[kTileBytes];
  uint8_t k[kStages][kTileBytes];
  uint8_t v[kStages][kTileBytes];
  uint64_t q_full;
  uint64_t k_full[kStages];
  uint64_t k_empty[kStages];
  uint64_t v_full[kStages];
  uint64_t v_empty[kStages];
  uint64_t s_full[2];   // S_j in TMEM buffer j % 2 is ready (tcgen05.commit)
  uint64_t p_ready[2];  // softmax done with buffer j % 2: decision taken, P written, O rescaled
  uint64_t o_done;      // the last issued P V has completed
  uint64_t drain;       // all MMAs of the CTA have completed
  uint32_t tmem_base;
  uint32_t skip_flag[2];
  uint32_t quit[2];     // softmax warps leave the loop together (one slot per iteration parity)
  uint32_t abort;       // some role gave up waiting
};
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;  // + slack to align the base to 1024 B

struct FwdParams {
  int B, H, Sq, Sk, nQ, nK;
  float scale_log2;   // scale * log2(e)
  float log2_lambda;  // log2(factor / Sk); -inf when factor == 0
  __nv_bfloat16* o;
  float* lse;
  uint32_t* skip_counts;
  uint8_t* skip_mask;
};

// Bounded wait on an mbarrier phase. Gives up after kWaitTimeoutNs, or at once
// when another role has given up (unless `respect_abort` is false); on a
// timeout it records `site` in the device error word and raises the CTA abort flag.
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
        *abort = 1u;
        atomicOr(&g_error_word, site);
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
__device__ __forceinline__ void run_producer(Smem& sm, const CUtensorMap* tq, const CUtensorMap* tk,
                                             const CUtensorMap* tv, const FwdParams& p, int b, int h,
                                             int qt) {
  volatile uint32_t* abort = &sm.abort;
  prefetch_tmap(tq);
  prefetch_tmap(tk);
  prefetch_tmap(tv);
  const uint32_t q_full = smem_u32(&sm.q_full);
  const uint32_t qs = smem_u32(sm.q);
  mbar_arrive_expect_tx(q_full, kTileBytes);
  tma_load_4d(qs, tq, q_full, 0, h, qt * kTile, b);
  tma_load_4d(qs + kHalfBytes, tq, q_full, 64, h, qt * kTile, b);

  int k_issued[kStages] = {0, 0};  // copies issued per stage
  int v_issued[kStages] = {0, 0};
  for (int j = 0; j < p.nK; ++j) {
    const int st = j & 1;
    const uint32_t empty_parity = ((j >> 1) + 1) & 1;  // completion j/2 - 1 of the empty barrier
    if (j >= kStages && !wait_bar(smem_u32(&sm.k_empty[st]), empty_parity, abort, kErrProducer)) break;
    const uint32_t kf = smem_u32(&sm.k_full[st]);
    const uint32_t ks = smem_u32(sm.k[st]);
    mbar_arrive_expect_tx(kf, kTileBytes);
    tma_load_4d(ks, tk, kf, 0, h, j * kTile, b);
    tma_load_4d(ks + kHalfBytes, tk, kf, 64, h, j * kTile, b);
    ++k_issued[st];
    if (j >= kStages && !wait_bar(smem_u32(&sm.v_empty[st]), empty_parity, abort, kErrProducer)) break;
    const uint32_t vf = smem_u32(&sm.v_full[st]);
    const uint32_t vs = smem_u32(sm.v[st]);
    mbar_arrive_expect_tx(vf, kTileBytes);
    tma_load_4d(vs, tv, vf, 0, h, j * kTile, b);
    tma_load_4d(vs + kHalfBytes, tv, vf, 64, h, j * kTile, b);
    ++v_issued[st];
  }
  // Every copy this thread issued lands before the CTA may exit (immediate on the normal
  // path, where the consumers have already waited for all of them).
  for (int st = 0; st < kStages; ++st) {
    if (k_issued[st] > 0) wait_bar(smem_u32(&sm.k_full[st]), (k_issued[st] - 1) & 1, abort, kErrDrain, false, kDrainTimeoutNs);
    if (v_issued[st] > 0) wait_bar(smem_u32(&sm.v_full[st]), (v_issued[st] - 1) & 1, abort, kErrDrain, false, kDrainTimeoutNs);
  }
  wait_bar(q_full, 0, abort, kErrDrain, false, kDrainTimeoutNs);
}

// ------------------------------------------------------------------ MMA issuer
__device__ __forceinline__ void run_mma(Smem& sm, uint32_t tmem, const FwdParams& p) {
  volatile uint32_t* abort = &sm.abort;
  constexpr uint32_t kIdescQK = idesc_bf16_f32(kTile, kTile, false);     // K tile is K-major
  constexpr uint32_t kIdescPV = idesc_bf16_f32(kTile, kHeadDim, true);   // V tile is MN-major
  const uint32_t qs = smem_u32(sm.q);

  // S = Q K^T: 8 steps of K = 16 features. Q and K tiles are two 64-feature halves of
  // 128-B swizzled rows; a step advances 32 B inside a half (SBO = 8 rows x 128 B).
  auto issue_qk = [&](uint32_t d_tmem, uint32_t ks) {
#pragma unroll
    for (int kk = 0; kk < kHeadDim / 16; ++kk) {
      const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
      mma_ss(d_tmem, smem_desc_sw128(qs + off, 16, 1024), smem_desc_sw128(ks + off, 16, 1024),
             kIdescQK, kk > 0 ? 1u : 0u);
    }
  };
  // O (+)= P V: 8 steps of K = 16 keys. P sits in TMEM (2 bf16 per column, 8 columns
  // per step). V rows are keys: a step advances 16 rows = 2 KiB; the two 64-feature
  // halves are LBO = 16 KiB apart, 8-row groups SBO = 1 KiB apart.
  auto issue_pv = [&](uint32_t p_tmem, uint32_t vs, bool accumulate) {
#pragma unroll
    for (int kk = 0; kk < kTile / 16; ++kk) {
      mma_ts(tmem + kColO, p_tmem + kk * 8, smem_desc_sw128(vs + kk * 2048, kHalfBytes, 1024),
             kIdescPV, (accumulate || kk > 0) ? 1u : 0u);
    }
  };

  int pv_issued = 0;
  bool ok = wait_bar(smem_u32(&sm.q_full), 0, abort, kErrMma) &&
            wait_bar(smem_u32(&sm.k_full[0]), 0, abort, kErrMma);
  if (ok) {
    tc_fence_after();
    issue_qk(tmem + col_s(0), smem_u32(sm.k[0]));
    tc_commit(smem_u32(&sm.s_full[0]));
    tc_commit(smem_u32(&sm.k_empty[0]));
    for (int j = 0; j < p.nK; ++j) {
      if (j + 1 < p.nK) {
        // Buffer (j+1) % 2 last held tile j-1, whose P V (if any) was issued before this
        // point; tcgen05.mma executes in issue order, so overwriting it is safe.
        const int st = (j + 1) & 1;
        if (!wait_bar(smem_u32(&sm.k_full[st]), ((j + 1) >> 1) & 1, abort, kErrMma)) break;
        tc_fence_after();
        issue_qk(tmem + col_s(st), smem_u32(sm.k[st]));
        tc_commit(smem_u32(&sm.s_full[st]));
        tc_commit(smem_u32(&sm.k_empty[st]));
      }
      const int sb = j & 1;
      const uint32_t parity = (j >> 1) & 1;
      if (!wait_bar(smem_u32(&sm.p_ready[sb]), parity, abort, kErrMma)) break;
      tc_fence_after();
      const uint32_t skip = *reinterpret_cast<volatile uint32_t*>(&sm.skip_flag[sb]);
      if (!wait_bar(smem_u32(&sm.v_full[sb]), parity, abort, kErrMma)) break;
      if (!skip) {
        tc_fence_after();
        issue_pv(tmem + col_s(sb), smem_u32(sm.v[sb]), pv_issued > 0);
        tc_commit(smem_u32(&sm.o_done));
        tc_commit(smem_u32(&sm.v_empty[sb]));
        ++pv_issued;
      } else {
        mbar_arrive(smem_u32(&sm.v_empty[sb]));  // V_j was loaded but is not needed
      }
    }
  }
  // Every MMA this thread issued completes before TMEM is released.
  tc_commit(smem_u32(&sm.drain));
  wait_bar(smem_u32(&sm.drain), 0, abort, kErrDrain, false, kDrainTimeoutNs);
}

// ------------------------------------------------------------------ softmax + epilogue
__device__ __forceinline__ void run_softmax(Smem& sm, uint32_t tmem, const FwdParams& p, int b,
                                            int h, int qt) {
  volatile uint32_t* abort = &sm.abort;
  volatile uint32_t* quit = sm.quit;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int row = threadIdx.x;  // query row inside the tile == TMEM lane
  const int q_row = qt * kTile + row;
  const bool row_valid = q_row < p.Sq;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t t_o = tmem + lane_base + kColO;
  const size_t mask_base =
      p.skip_mask ? ((static_cast<size_t>(b) * p.H + h) * p.nQ + qt) * static_cast<size_t>(p.nK) : 0;

  float m_run = -INFINITY;  // running max of scaled scores (log2 units), kept tiles only
  float m_use = -INFINITY;  // exponent reference of l and O (trails m_run by <= 8)
  float l = 0.f;
  int pv_count = 0;
  uint32_t skipped = 0;
  bool failed = false;
  bool left_early = false;

  for (int j = 0; j < p.nK; ++j) {
    const int sb = j & 1;
    const uint32_t t_s = tmem + lane_base + col_s(sb);
    bool pass = true;
    float s[kTile];
    float tm2 = 0.f;
    if (!failed) {
      const bool ok = wait_bar(smem_u32(&sm.s_full[sb]), (j >> 1) & 1, abort, kErrSoftmax);
      failed = !__all_sync(0xffffffffu, ok);
    }
    if (!failed) {
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < kTile / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(t_s + c * 32, r);
#pragma unroll
        for (int t = 0; t < 32; ++t) s[c * 32 + t] = __uint_as_float(r[t]);
      }
      const int valid_keys = p.Sk - j * kTile;
      if (valid_keys < kTile) {
#pragma unroll
        for (int c = 0; c < kTile; ++c)
          if (c >= valid_keys) s[c] = -INFINITY;
      }
      float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
      for (int c = 4; c < kTile; c += 4) {
        mx0 = fmaxf(mx0, s[c]);
        mx1 = fmaxf(mx1, s[c + 1]);
        mx2 = fmaxf(mx2, s[c + 2]);
        mx3 = fmaxf(mx3, s[c + 3]);
      }
      tm2 = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * p.scale_log2;
      // The skip test for this row; rows past Sq do not exist and always pass.
      pass = !row_valid || (tm2 - m_run < p.log2_lambda);
    } else {
      quit[sb] = 1u;
    }
    const bool skip = bar_and<1, kSoftmaxThreads>(pass);
    if (quit[sb]) {  // written only before this barrier: every softmax thread sees the same value
      left_early = true;
      break;
    }
    if (threadIdx.x == 0 && p.skip_mask) p.skip_mask[mask_base + j] = skip ? 1 : 0;

    if (skip) {
      if (threadIdx.x == 0) {
        sm.skip_flag[sb] = 1u;
        ++skipped;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.p_ready[sb]));
      continue;
    }

    // Kept tile: online-softmax update.
    const float m_new = fmaxf(m_run, tm2);
    m_run = m_new;
    float alpha = 1.f;
    if (m_new - m_use > kRescaleThreshold) {
      alpha = ex2_approx(m_use - m_new);  // 0 for the first kept tile
      m_use = m_new;
    }
    const float neg_ref = -m_use;
    // P (bf16, keys 2c and 2c+1 in column c) overwrites the first 64 columns of S_j,
    // written in two halves of 32 columns as it is produced.
    float sum0 = 0.f, sum1 = 0.f, sum2 = 0.f, sum3 = 0.f;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      uint32_t pk[32];
#pragma unroll
      for (int c = 0; c < 32; c += 2) {
        const int k0 = half * 64 + 2 * c;
        const float p0 = ex2_approx(fmaf(s[k0 + 0], p.scale_log2, neg_ref));
        const float p1 = ex2_approx(fmaf(s[k0 + 1], p.scale_log2, neg_ref));
        const float p2 = ex2_approx(fmaf(s[k0 + 2], p.scale_log2, neg_ref));
        const float p3 = ex2_approx(fmaf(s[k0 + 3], p.scale_log2, neg_ref));
        sum0 += p0;
        sum1 += p1;
        sum2 += p2;
        sum3 += p3;
        pk[c] = pack_bf16(p0, p1);
        pk[c + 1] = pack_bf16(p2, p3);
      }
      tmem_st32(t_s + half * 32, pk);
    }
    tmem_st_wait();
    l = l * alpha + ((sum0 + sum1) + (sum2 + sum3));
    if (pv_count > 0) {
      // The previous P V must be finished before O is touched (and before the next is issued).
      const bool ok = wait_bar(smem_u32(&sm.o_done), (pv_count - 1) & 1, abort, kErrSoftmax);
      failed = !__all_sync(0xffffffffu, ok);
      if (!failed && __any_sync(0xffffffffu, alpha != 1.f)) {
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < kHeadDim / 32; ++c) {
          uint32_t r[32];
          tmem_ld32(t_o + c * 32, r);
#pragma unroll
          for (int t = 0; t < 32; ++t) r[t] = __float_as_uint(__uint_as_float(r[t]) * alpha);
          tmem_st32(t_o + c * 32, r);
        }
        tmem_st_wait();
      }
    }
    if (!failed) {
      if (threadIdx.x == 0) sm.skip_flag[sb] = 0u;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.p_ready[sb]));
    }
    ++pv_count;
  }

  if (!left_early && !failed && pv_count > 0) {
    const bool ok = wait_bar(smem_u32(&sm.o_done), (pv_count - 1) & 1, abort, kErrSoftmax);
    if (__all_sync(0xffffffffu, ok)) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      __nv_bfloat16* orow =
          p.o + ((static_cast<size_t>(b) * p.Sq + (row_valid ? q_row : 0)) * p.H + h) * kHeadDim;
#pragma unroll
      for (int c = 0; c < kHeadDim / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(t_o + c * 32, r);
        if (row_valid) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            uint4 w;
            w.x = pack_bf16(__uint_as_float(r[8 * t + 0]) * inv_l, __uint_as_float(r[8 * t + 1]) * inv_l);
            w.y = pack_bf16(__uint_as_float(r[8 * t + 2]) * inv_l, __uint_as_float(r[8 * t + 3]) * inv_l);
            w.z = pack_bf16(__uint_as_float(r[8 * t + 4]) * inv_l, __uint_as_float(r[8 * t + 5]) * inv_l);
            w.w = pack_bf16(__uint_as_float(r[8 * t + 6]) * inv_l, __uint_as_float(r[8 * t + 7]) * inv_l);
            dst[t] = w;
          }
        }
      }
      if (row_valid && p.lse)
        p.lse[(static_cast<size_t>(b) * p.H + h) * p.Sq + q_row] = (m_use + log2f(l)) * kLn2;
    }
  }
  if (threadIdx.x == 0 && p.skip_counts && skipped)
    atomicAdd(&p.skip_counts[static_cast<size_t>(b) * p.H + h], skipped);
}

__global__ void __launch_bounds__(kThreads, 1)
    blasst_fwd_sm103a(const __grid_constant__ CUtensorMap tmap_q,
                      const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v, const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                      ~static_cast<uintptr_t>(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm.q_full), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&sm.k_full[s]), 1);
      mbar_init(smem_u32(&sm.k_empty[s]), 1);
      mbar_init(smem_u32(&sm.v_full[s]), 1);
      mbar_init(smem_u32(&sm.v_empty[s]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm.s_full[i]), 1);
      mbar_init(smem_u32(&sm.p_ready[i]), kSoftmaxWarps);
      sm.skip_flag[i] = 0u;
      sm.quit[i] = 0u;
    }
    mbar_init(smem_u32(&sm.o_done), 1);
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
  const uint32_t tmem = sm.tmem_base;

  if (warp == kLoadWarp) {
    if (lane == 0) run_producer(sm, &tmap_q, &tmap_k, &tmap_v, p, b, h, qt);
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0) run_mma(sm, tmem, p);
    __syncwarp();
  } else {
    run_softmax(sm, tmem, p, b, h, qt);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
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

// [B, S, H, 128] bf16 viewed as a 4-D tensor (d, H, S, B); boxes of 64 features x 1 head x
// 128 tokens x 1 batch, 128-byte swizzled. Tokens past S read as zero.
bool encode_bshd(CUtensorMap* map, const void* base, int B, int S, int H) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(S), static_cast<cuuint64_t>(B)};
  const cuuint64_t row = static_cast<cuuint64_t>(kHeadDim) * 2;
  const cuuint64_t strides[3] = {row, row * static_cast<cuuint64_t>(H),
                                 row * static_cast<cuuint64_t>(H) * static_cast<cuuint64_t>(S)};
  const cuuint32_t box[4] = {64, 1, static_cast<cuuint32_t>(kTile), 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
  if (cudaFuncSetAttribute(blasst_fwd_sm103a, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSmemBytes)) != cudaSuccess) {
    cudaGetLastError();
    return BLASST_ERR_LAUNCH;
  }
  g_dev_state[dev] = 1;
  return BLASST_OK;
}

bool aligned(const void* ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; }

}  // namespace
}  // namespace blasst

extern "C" blasst_status blasst_attn_fwd(const void* q, const void* k, const void* v, void* o,
                                         float* lse, int B, int H, int Sq, int Sk, int d,
                                         float scale, float factor, struct CUstream_st* stream,
                                         uint32_t* skip_counts, uint8_t* skip_mask_dbg) {
  using namespace blasst;
  // ---- argument checks: no CUDA call happens before all of them pass
  if (!q || !k || !v || !o) return BLASST_ERR_INVALID_ARG;
  if (B <= 0 || H <= 0 || Sq <= 0 || Sk <= 0 || B > 65535 || H > 65535) return BLASST_ERR_INVALID_ARG;
  if (d != kHeadDim) return BLASST_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return BLASST_ERR_INVALID_ARG;
  if (!std::isfinite(factor) || !(factor >= 0.f)) return BLASST_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
    return BLASST_ERR_INVALID_ARG;
  if (lse && !aligned(lse, 4)) return BLASST_ERR_INVALID_ARG;
  // byte strides of the 4-D views must stay below 2^40 (TMA limit)
  const double batch_stride = 256.0 * H * static_cast<double>(Sq > Sk ? Sq : Sk);
  if (batch_stride >= 1099511627776.0) return BLASST_ERR_INVALID_ARG;

  const blasst_status ds = prepare_device();
  if (ds != BLASST_OK) return ds;

  CUtensorMap tq, tk, tv;
  if (!encode_bshd(&tq, q, B, Sq, H) || !encode_bshd(&tk, k, B, Sk, H) ||
      !encode_bshd(&tv, v, B, Sk, H))
    return BLASST_ERR_LAUNCH;

  FwdParams p{};
  p.B = B;
  p.H = H;
  p.Sq = Sq;
  p.Sk = Sk;
  p.nQ = (Sq + kTile - 1) / kTile;
  p.nK = (Sk + kTile - 1) / kTile;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.log2_lambda = factor > 0.f ? static_cast<float>(std::log2(static_cast<double>(factor) / Sk))
                               : -INFINITY;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.skip_counts = skip_counts;
  p.skip_mask = skip_mask_dbg;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (skip_counts &&
      cudaMemsetAsync(skip_counts, 0, sizeof(uint32_t) * static_cast<size_t>(B) * H, st) != cudaSuccess) {
    cudaGetLastError();
    return BLASST_ERR_LAUNCH;
  }
  void* args[] = {&tq, &tk, &tv, &p};
  const cudaError_t e = cudaLaunchKernel(reinterpret_cast<const void*>(blasst_fwd_sm103a),
                                         dim3(p.nQ, H, B), dim3(kThreads), args, kSmemBytes, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return BLASST_ERR_LAUNCH;
  }
  return BLASST_OK;
}

extern "C" const char* blasst_status_string(blasst_status s) {
  switch (s) {
    case BLASST_OK: return "ok";
    case BLASST_ERR_INVALID_ARG: return "invalid argument";
    case BLASST_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
    case BLASST_ERR_LAUNCH: return "CUDA launch or set-up failure";
    case BLASST_ERR_TIMEOUT: return "a device-side wait timed out";
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

extern "C" int blasst_version(void) { return 100; }
