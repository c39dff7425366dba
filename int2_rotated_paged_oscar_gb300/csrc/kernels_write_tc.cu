// Prefill / extend write of the OSCAR INT2 cache on the 5th-generation tensor
// cores (tcgen05 + TMEM), for BF16 inputs and a dense rotation R.
//
// Source: OSCAR technical summary (gist.science), section 2.2 B -- history is
// stored in INT2 after the fixed rotation and clipping; arXiv abstract -- fused
// write kernel.  The rotation y = x R of a tile of 128 (token, kv head) rows is
// a 128 x D x D GEMM:
//   A = the rows, BF16 as received, staged by TMA with 128-byte swizzling;
//   B = R split exactly into three BF16 planes R = R1 + R2 + R3 (R1 = bf16(R),
//       R2 = bf16(R - R1), R3 = bf16(R - R1 - R2): 3 x 8 significant bits cover
//       float32's 24), held transposed (K-major) in shared memory for the
//       whole launch;
//   D = float32 in tensor memory: per tile two partial accumulators (the small
//       planes and the first half of K of R1; the second half of K of R1), added in
//       float32 by the epilogue, and two such buffers so that the MMAs of one tile
//       overlap the epilogue of the previous one.
// Products of BF16 values are exact and accumulate in float32, so y carries
// float32-level error like the CUDA-core path (not the same rounding).
// Hadamard-only rotation (R = H_Had P_br / sqrt(D), the data-oblivious baseline of
// section 2.2 A): R sqrt(D) has entries +-1, exact in one BF16 plane built in the kernel,
// (H P_br)[i][j] = (-1)^popcount(i & br(j)) for the natural-order Sylvester H and the
// bit reversal br; one accumulator per tile, scaled by 1/sqrt(D) in the epilogue.
// Epilogue: thread t of the four epilogue warps owns row t of the tile (TMEM lane
// t): it reads the row group by group (32 columns), clips, finds min/max, forms
// the BF16 zero and scale, rounds the codes (reciprocal multiply) and packs the
// K or V code row in registers.  Window rows (sink / recent) are copied to the
// BF16 slab unrotated.
// Roles: the epilogue warps (per TMEM buffer and per column half of the row, one warp
// per TMEM lane quadrant), then one producer warp (TMA, MMA issue, TMEM allocation).
// Every mbarrier wait is bounded by %globaltimer; a timeout flags the status
// word and the CTA stops issuing work.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "oscar_internal.h"

namespace oscar {
namespace {

constexpr int kTileM = 128;
// Epilogue warps: for each of the two TMEM buffers and each column half of the row,
// four warps (one per TMEM lane quadrant); the producer warp comes after them.
#ifndef OSCAR_WRITE_HALVES
#define OSCAR_WRITE_HALVES 1
#endif
template <int D> __host__ __device__ constexpr int epi_halves() { return D == 128 ? OSCAR_WRITE_HALVES : 1; }
template <int D> __host__ __device__ constexpr int epi_warps() { return 2 * epi_halves<D>() * 4; }
template <int D> __host__ __device__ constexpr int tc_threads() { return (epi_warps<D>() + 1) * 32; }

#include "tc_common.cuh"

// ------------------------------------------------------------------ shared memory plan
template <int D, bool HAD>
struct TcPlan {
  static constexpr int PLANES = HAD ? 1 : 3;         // BF16 planes of R^T
  static constexpr int KCH = D / 64;                 // 128-byte K chunks per row
  static constexpr int NS = 4;                       // row-tile stages in flight
  static constexpr int A_BYTES = kTileM * D * 2;     // one A stage
  static constexpr int B_PLANE = D * D * 2;          // one BF16 plane of R^T
  static constexpr int A_OFF = PLANES * B_PLANE;     // multiple of 1024
  static constexpr int BAR_OFF = A_OFF + NS * A_BYTES;
  static constexpr int NBARS = 2 * NS + 5;           // a_full[NS], a_empty[NS], acc_full[2], acc_empty[2], r_full
  static_assert((NS - 2) * A_BYTES >= D * D * 4, "R (float32) is staged in A stages 2 .. NS-1");
  static constexpr int BYTES = BAR_OFF + NBARS * 8 + 16;
  static constexpr int SMEM = BYTES + 1024;          // slack for the 1024-byte alignment of the base
  // per tile buffer two float32 accumulators of D columns (see the MMA order; one with the
  // Hadamard plane); two buffers
  static constexpr uint32_t ACC_COLS = HAD ? D : 2 * D;
  static constexpr uint32_t TMEM_COLS = 2 * ACC_COLS;
};

__device__ __forceinline__ uint16_t bf16_bits_rn(float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<const uint16_t*>(&h);
}

// Clip, quantise and pack group gi (32 channels, this thread's row) into the code
// words and the (scale, zero) word.  The group's min and max are clipped (clipping
// is monotonic, so they equal those of the clipped values); the codes are
// clamp(rne((clip(y) - z) / s), 0, 3) computed as y * (1/s) - z/s clamped to the
// images of the clip range and to [0, 3] in float, then rounded to nearest-even by
// adding 1.5 * 2^23, whose float pattern carries the code in its low bits.  The code
// words accumulate pattern << shift with one integer multiply-add per code; the
// caller starts each word at minus the patterns' constant part (code_bias).
constexpr float kRoundMagic = 12582912.0f;     // 1.5 * 2^23
constexpr uint32_t kRoundBits = 0x4B400000u;   // its float pattern
template <int D, bool IS_V>
__device__ __forceinline__ void quant_group(const float (&y)[32], int gi, float clip, uint32_t (&words)[D / 16],
                                            uint32_t& szw) {
  float mn = y[0], mx = y[0];
#pragma unroll
  for (int j = 1; j < 32; ++j) {
    mn = fminf(mn, y[j]);
    mx = fmaxf(mx, y[j]);
  }
  mn = fminf(fmaxf(mn, -clip), clip);
  mx = fminf(fmaxf(mx, -clip), clip);
  const uint16_t zb = bf16_bits_rn(mn);
  const uint16_t sb = bf16_bits_rn((mx - mn) / 3.0f);
  const float z = __uint_as_float(static_cast<uint32_t>(zb) << 16);
  const float sc = __uint_as_float(static_cast<uint32_t>(sb) << 16);
  const float inv = sc > 0.f ? __frcp_rn(sc) : 0.f;  // s = 0: every code 0
  const float zinv = -z * inv;
  // y -> y * inv - z * inv is monotonic, so clamping it to the images of -clip and
  // clip is the same as clipping y first; then clamp to [0, 3].  The image of clip is
  // below 0 when z, the group minimum rounded to BF16, lands above a clip that BF16
  // cannot represent and the group spans less than that rounding: every code is then
  // 0, and t_hi must not go below 0 (a negative code would borrow from its neighbours
  // in the packed word).  t_lo above 3 needs no care: t_hi <= 3 wins the clamp.
  const float t_lo = fmaxf(fmaf(-clip, inv, zinv), 0.f);
  const float t_hi = fmaxf(fminf(fmaf(clip, inv, zinv), 3.f), 0.f);
  // the code argument and the rounding add in float32 pairs (two IEEE operations each,
  // the same results as the scalar forms)
  const float2 inv2 = make_float2(inv, inv), zinv2 = make_float2(zinv, zinv);
  const float2 mag2 = make_float2(kRoundMagic, kRoundMagic);
  float tp[32];
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const float2 t2 = __ffma2_rn(make_float2(y[j], y[j + 1]), inv2, zinv2);
    const float2 c2 = make_float2(fminf(fmaxf(t2.x, t_lo), t_hi), fminf(fmaxf(t2.y, t_lo), t_hi));
    const float2 p2 = __fadd2_rn(c2, mag2);
    tp[j] = p2.x;
    tp[j + 1] = p2.y;
  }
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const uint32_t pat = __float_as_uint(tp[j]);  // kRoundBits + code
    const int c = 32 * gi + j;
    int word, shift;
    if constexpr (!IS_V) {
      // K row: word tig*(D/64) + w holds slot x at bits 2x (channel c) and 16 + 2x (c + 1)
      const int tig = (j & 7) >> 1, e = j & 1, h = (j >> 3) & 1, kt = j >> 4;
      word = tig * (D / 64) + (gi >> 1);
      shift = 16 * e + 2 * (4 * (gi & 1) + 2 * kt + h);
    } else {
      // V row: half-word hw = (D/64)(c mod 8) + c/64 holds channel c at bits 2 ((c mod 64) / 8)
      const int hw = (D / 64) * (c & 7) + (c >> 6);
      word = hw >> 1;
      shift = 16 * (hw & 1) + 2 * ((c & 63) >> 3);
    }
    words[word] += pat << shift;
  }
  szw = static_cast<uint32_t>(sb) | (static_cast<uint32_t>(zb) << 16);
}

// Sum over the codes of channels [c_lo, c_hi) of a row of kRoundBits << shift, per
// word (the constant part of the accumulated patterns), for K or V rows;
// constant-folded when unrolled.
template <int D, bool IS_V>
__device__ __forceinline__ uint32_t code_bias(int word, int c_lo, int c_hi) {
  uint32_t acc = 0;
#pragma unroll
  for (int c = 0; c < D; ++c) {
    if (c < c_lo || c >= c_hi) continue;
    const int gi = c / 32, j = c % 32;
    int w, sh;
    if constexpr (!IS_V) {
      const int tig = (j & 7) >> 1, e = j & 1, h = (j >> 3) & 1, kt = j >> 4;
      w = tig * (D / 64) + (gi >> 1);
      sh = 16 * e + 2 * (4 * (gi & 1) + 2 * kt + h);
    } else {
      const int hw = (D / 64) * (c & 7) + (c >> 6);
      w = hw >> 1;
      sh = 16 * (hw & 1) + 2 * ((c & 63) >> 3);
    }
    if (w == word) acc += kRoundBits << sh;
  }
  return acc;
}

template <int D, bool HAD>
__global__ void __launch_bounds__(tc_threads<D>(), 1) write_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                                                 const __grid_constant__ CUtensorMap tmap_v,
                                                                 WriteArgs a) {
  using L = TcPlan<D, HAD>;
  constexpr int kEpiWarps = epi_warps<D>();
  constexpr int HALVES = epi_halves<D>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool is_v = blockIdx.y == 1;
  const Geom& g = a.g;
  uint8_t* bsm = smem;
  uint8_t* asm_ = smem + L::A_OFF;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::BAR_OFF);
  uint64_t* a_full = bars;
  uint64_t* a_empty = bars + L::NS;
  uint64_t* acc_full = bars + 2 * L::NS;
  uint64_t* acc_empty = acc_full + 2;
  uint64_t* r_full = acc_empty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + L::NBARS);
  // Work items are tiles of kTileM rows.  One rotation per layer: rows r = token * Hkv + h
  // of the whole call, tile i covering rows [kTileM i, kTileM (i + 1)), split over the CTAs.
  // A rotation per kv head: CTA x keeps kv head x mod Hkv (and that head's R planes) and
  // takes the tiles of 128 consecutive tokens of that head, loaded by a 3-D tensor map.
  const int hsel = g.rph ? (int)blockIdx.x % g.Hkv : 0;
  const int cta_k = g.rph ? (int)blockIdx.x / g.Hkv : (int)blockIdx.x;
  const int n_ctas = g.rph ? (int)gridDim.x / g.Hkv : (int)gridDim.x;
  const long long rows = g.rph ? (long long)a.total_tokens : (long long)a.total_tokens * g.Hkv;
  const int tiles = (int)((rows + kTileM - 1) / kTileM);

  // R^T as three BF16 planes, K-major with the 128-byte swizzle (row n = column n of R).
  // R (float32, D x D) arrives by one bulk copy in A stages 2 .. NS-1, which the row tiles use
  // only after the planes are built; the producer thread requests this CTA's first two row
  // tiles (stages 0 and 1) at the same time, so their loads overlap the plane build.
  const float* R = (is_v ? a.R_V : a.R_K) + (size_t)hsel * g.rot_stride();
  const float* Rs = reinterpret_cast<const float*>(asm_ + 2 * L::A_BYTES);
  const bool producer = threadIdx.x == kEpiWarps * 32;
  const int n_mine = cta_k < tiles ? (tiles - 1 - cta_k) / n_ctas + 1 : 0;  // this CTA's row tiles
  const CUtensorMap* tmap = is_v ? &tmap_v : &tmap_k;
  auto load = [&](int i) {  // producer: tile i of this CTA into stage i % NS
    const int st = i % L::NS;
    mbar_arrive_expect_tx(&a_full[st], L::A_BYTES);
    const int tile = cta_k + i * n_ctas;
#pragma unroll
    for (int c = 0; c < L::KCH; ++c) {
      if (g.rph)
        tma_load_3d_tc(asm_ + st * L::A_BYTES + c * kTileM * 128, tmap, 64 * c, hsel, tile * kTileM, &a_full[st]);
      else
        tma_load_2d_tc(asm_ + st * L::A_BYTES + c * kTileM * 128, tmap, 64 * c, tile * kTileM, &a_full[st]);
    }
  };
  const int n_early = n_mine < 2 ? n_mine : 2;
  if (producer) {
    for (int i = 0; i < L::NS; ++i) {
      mbar_init(&a_full[i], 1);
      mbar_init(&a_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_empty[i], (kEpiWarps / 2) * 32);  // every epilogue warp of that buffer
    }
    mbar_init(r_full, 1);
    fence_barrier_init();
    if constexpr (!HAD) {
      mbar_arrive_expect_tx(r_full, D * D * sizeof(float));
      bulk_g2s(asm_ + 2 * L::A_BYTES, R, D * D * sizeof(float), r_full);
    }
    for (int i = 0; i < n_early; ++i) load(i);
  }
  __syncthreads();
  const bool r_ok = HAD || __syncthreads_and(mbar_wait_bounded(r_full, 0, a.status));
  if (!r_ok && producer) {  // drain every copy in flight before the CTA ends
    (void)mbar_wait_bounded(r_full, 0, nullptr);
    for (int i = 0; i < n_early; ++i) (void)mbar_wait_bounded(&a_full[i], 0, nullptr);
  }
  if constexpr (HAD) {
    // the +-1 plane: item = (n, k-octet); column n of H P_br is column br(n) of H
    constexpr int LOGD = D == 128 ? 7 : 6;
    for (int item = threadIdx.x; item < D * D / 8; item += blockDim.x) {
      const int n = item % D, k0 = (item / D) * 8;
      const uint32_t brn = __brev((uint32_t)n) >> (32 - LOGD);
      uint32_t pk[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t lo = (__popc((uint32_t)(k0 + 2 * q) & brn) & 1) ? 0xBF80u : 0x3F80u;
        const uint32_t hi = (__popc((uint32_t)(k0 + 2 * q + 1) & brn) & 1) ? 0xBF80u : 0x3F80u;
        pk[q] = lo | (hi << 16);
      }
      *reinterpret_cast<uint4*>(bsm + sw128_offset(n, k0, D)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
    }
  }
  // item = (n, k-octet): 8 consecutive k of column n, contiguous in the swizzled row
  for (int item = threadIdx.x; !HAD && r_ok && item < D * D / 8; item += blockDim.x) {
    const int n = item % D, k0 = (item / D) * 8;
    uint32_t pk[3][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t lo[3], hi[3];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float r = Rs[(k0 + 2 * q + e) * D + n];
        const __nv_bfloat16 p1 = __float2bfloat16_rn(r);
        const float r1 = r - __bfloat162float(p1);
        const __nv_bfloat16 p2 = __float2bfloat16_rn(r1);
        const __nv_bfloat16 p3 = __float2bfloat16_rn(r1 - __bfloat162float(p2));
        const uint32_t b1 = *reinterpret_cast<const uint16_t*>(&p1), b2 = *reinterpret_cast<const uint16_t*>(&p2),
                       b3 = *reinterpret_cast<const uint16_t*>(&p3);
        (e ? hi : lo)[0] = b1;
        (e ? hi : lo)[1] = b2;
        (e ? hi : lo)[2] = b3;
      }
#pragma unroll
      for (int p = 0; p < 3; ++p) pk[p][q] = lo[p] | (hi[p] << 16);
    }
    const uint32_t off = sw128_offset(n, k0, D);
#pragma unroll
    for (int p = 0; p < 3; ++p)
      *reinterpret_cast<uint4*>(bsm + p * L::B_PLANE + off) = make_uint4(pk[p][0], pk[p][1], pk[p][2], pk[p][3]);
  }
  if (warp == kEpiWarps) tmem_alloc(tmem_slot, L::TMEM_COLS);
  // the planes were written and R read by ordinary accesses; the MMAs read the planes and the
  // row-tile loads overwrite R through the async proxy
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kEpiWarps) {
    // ---------------- producer: TMA of the row tiles (NS ahead), MMA issue (one thread)
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kTileM, D);
      const uint32_t b_base = smem_u32(bsm);
      const int n_run = r_ok ? n_mine : 0;
      for (int i = n_early; i < L::NS && i < n_run; ++i) load(i);  // stages 2 .. NS-1, free of R now
      int i = 0;
      for (; i < n_run; ++i) {
        const int st = i % L::NS;
        const int s = i & 1;  // TMEM buffer
        if (!mbar_wait_bounded(&a_full[st], (uint32_t)(i / L::NS) & 1, a.status)) break;
        if (i >= 2 && !mbar_wait_bounded(&acc_empty[s], (uint32_t)((i >> 1) - 1) & 1, a.status)) break;
        tc_fence_after();
        const uint32_t a_base = smem_u32(asm_ + st * L::A_BYTES);
        const uint32_t acc0 = tmem + (uint32_t)(s * L::ACC_COLS), acc1 = acc0 + (uint32_t)D;
        if constexpr (HAD) {
          // one exact +-1 plane, one accumulator
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t ak = (uint32_t)((kk >> 2) * kTileM * 128 + (kk & 3) * 32);
            const uint32_t bk = (uint32_t)((kk >> 2) * D * 128 + (kk & 3) * 32);
            tc_mma_bf16(acc0, smem_desc_sw128(a_base + ak), smem_desc_sw128(b_base + bk), idesc, kk ? 1u : 0u);
          }
        } else {
          // Accuracy: each MMA rounds its float32 accumulation once, relative to the running
          // magnitude.  The small planes R3, R2 go first (into acc0, still small), then the
          // main plane R1 over the first half of K into acc0 and over the second half into
          // acc1; the epilogue adds acc0 + acc1 in float32.
#pragma unroll
          for (int pp = 0; pp < L::PLANES; ++pp) {
            const int p = L::PLANES - 1 - pp;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const bool second = p == 0 && kk >= D / 32;
              const uint32_t ak = (uint32_t)((kk >> 2) * kTileM * 128 + (kk & 3) * 32);
              const uint32_t bk = (uint32_t)(p * L::B_PLANE + (kk >> 2) * D * 128 + (kk & 3) * 32);
              const uint32_t first = (pp == 0 && kk == 0) || (p == 0 && kk == D / 32);
              tc_mma_bf16(second ? acc1 : acc0, smem_desc_sw128(a_base + ak), smem_desc_sw128(b_base + bk), idesc,
                          first ? 0u : 1u);
            }
          }
        }
        tc_commit(&a_empty[st]);
        tc_commit(&acc_full[s]);
        // refill the stage of the previous tile (its MMAs were issued one tile ago)
        if (i >= 1 && i - 1 + L::NS < n_run) {
          const int pst = (i - 1) % L::NS;
          if (!mbar_wait_bounded(&a_empty[pst], (uint32_t)((i - 1) / L::NS) & 1, a.status)) break;
          load(i - 1 + L::NS);
        }
      }
      // every MMA-completion arrival lands before the CTA may exit
      for (int j = (i > L::NS ? i - L::NS : 0); j < i; ++j)
        (void)mbar_wait_bounded(&a_empty[j % L::NS], (uint32_t)(j / L::NS) & 1, nullptr);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue: warp w reads TMEM lane quadrant w % 4, takes the tiles of
    // buffer eg = (w / 4) % 2 and the column half ch = w / 8 (groups [ch G/H, (ch+1) G/H));
    // thread t owns row t of the tile
    const int eg = (warp >> 2) & 1;
    const int ch = warp >> 3;
    const int t = (warp & 3) * 32 + lane;
    constexpr int GPH = D / 32 / HALVES;  // groups per half
    const float clip = is_v ? a.clip_V : a.clip_K;
    const void* src = is_v ? a.V : a.K;
    // the eviction launched before this kernel reads ring rows that the tiles' window rows
    // overwrite: every store waits for it (the set-up and the row-tile loads did not)
    pdl_wait();
    int i = eg;
    // this thread's request from its previous tile (rows advance, and a request spans many
    // tiles): tokens [c_lo, c_hi) of request c_b, first position c_t0; c_b < 0: none yet.  Kept
    // by the one-plane form only: the dense form's epilogue has no registers to spare for it
    // (168 a thread, the limit at nine warps; the four more spilled and made it slower).
    int c_b = -1, c_lo = 0, c_hi = 0, c_t0 = 0;
    for (int tile = cta_k + eg * n_ctas; r_ok && tile < tiles; tile += 2 * n_ctas, i += 2) {
      const int s = i & 1;
      const uint32_t u = (uint32_t)(i >> 1);
      // where this row goes: 1 = INT2 history slot, 2 = BF16 window slot, 0 = nowhere
      const long long r = (long long)tile * kTileM + t;
      int kind = 0, b = 0, pos = 0, h = 0, token = 0;
      if (r < rows) {
        token = g.rph ? static_cast<int>(r) : static_cast<int>(r / g.Hkv);
        h = g.rph ? hsel : static_cast<int>(r % g.Hkv);
        if (!HAD || c_b < 0 || token < c_lo || token >= c_hi) {
          int lo = 0, hi = a.batch - 1;  // request: largest b with cu_seqlens[b] <= token
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a.cu_seqlens[mid] <= token) lo = mid; else hi = mid - 1;
          }
          c_b = lo;
          c_lo = a.cu_seqlens[lo];
          c_hi = a.cu_seqlens[lo + 1];
          c_t0 = a.start_pos[lo];
        }
        b = c_b;
        const int t0 = c_t0;
        const int n1 = t0 + (c_hi - c_lo);
        pos = t0 + (token - c_lo);
        if (t0 < 0 || n1 > g.max_pages_per_req * g.P) {
          flag_error(a.status, kDevBadLen);
        } else {
          kind = (pos >= g.S && pos < n1 - g.W) ? 1 : 2;
        }
      }
      int page = -1, req = -1;  // looked up while the tile's MMAs run
      if (kind == 1) {
        const int lp = pos / g.P;
        if (lp < a.bt_stride && lp < g.max_pages_per_req) page = a.block_table[(size_t)b * a.bt_stride + lp];
      } else if (kind == 2) {
        req = a.req_slot[b];
      }
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&acc_full[s], u & 1, a.status))) break;
      tc_fence_after();
      // read this row's groups from TMEM, quantise and pack; CH (column half) and IS_V are
      // compile-time so that every code lands at a constant bit position
      auto quant_store = [&](auto ch_tag, auto v_tag) {
        constexpr int CH = decltype(ch_tag)::value;
        constexpr bool IS_V = decltype(v_tag)::value;
        constexpr int C_LO = CH * GPH * 32, C_HI = C_LO + GPH * 32;
        uint32_t words[D / 16];
        uint32_t szw[D / 32];
#pragma unroll
        for (int w = 0; w < D / 16; ++w) words[w] = 0u - code_bias<D, IS_V>(w, C_LO, C_HI);
        // a group's accumulators are read from TMEM while the previous group is quantised
        uint32_t r0[32], r1[HAD ? 1 : 32];
        (void)r1;
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(s * L::ACC_COLS);
        constexpr float kInvSqrtD = D == 64 ? 0.125f : 0.08838834764831845f;   // 1/sqrt(D) rounded to float32
        const float2 hscale = make_float2(kInvSqrtD, kInvSqrtD);
        auto load_group = [&](int gg) {
          tmem_ld32_nowait(lane_base + (uint32_t)(32 * gg), r0);
          if constexpr (!HAD) tmem_ld32_nowait(lane_base + (uint32_t)(32 * gg + D), reinterpret_cast<uint32_t(&)[32]>(r1));
        };
        load_group(CH * GPH);
#pragma unroll
        for (int gq = 0; gq < GPH; ++gq) {
          const int gi = CH * GPH + gq;
          tmem_wait_ld();
          float y[32];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float2 a2 = make_float2(__uint_as_float(r0[j]), __uint_as_float(r0[j + 1]));
            float2 s2;
            if constexpr (HAD) s2 = __fmul2_rn(a2, hscale);
            else s2 = __fadd2_rn(a2, make_float2(__uint_as_float(r1[j]), __uint_as_float(r1[j + 1])));
            y[j] = s2.x;
            y[j + 1] = s2.y;
          }
          if (gq + 1 < GPH) load_group(gi + 1);
          quant_group<D, IS_V>(y, gi, clip, words, szw[gi]);
        }
        tc_fence_before();
        mbar_arrive(&acc_empty[s]);  // this accumulator may be overwritten once every row is read
        if (kind != 1) return;
        if (page < 0 || page >= g.num_pages) {
          flag_error(a.status, kDevBadPage);
          return;
        }
        uint8_t* blk = a.pool + (((size_t)a.layer * g.num_pages + page) * g.Hkv + h) * g.block_bytes();
        uint8_t* crow = blk + (IS_V ? g.v_codes_off() : 0) + (size_t)(pos % g.P) * (D / 4);
        uint32_t* szp =
            reinterpret_cast<uint32_t*>(blk + (IS_V ? g.v_sz_off() : g.k_sz_off()) + (size_t)(pos % g.P) * (D / 8));
        if constexpr (HALVES == 1) {
          uint4* codes = reinterpret_cast<uint4*>(crow);
#pragma unroll
          for (int q = 0; q < D / 64; ++q)
            codes[q] = make_uint4(words[4 * q], words[4 * q + 1], words[4 * q + 2], words[4 * q + 3]);
#pragma unroll
          for (int gi = 0; gi < D / 32; ++gi) szp[gi] = szw[gi];
        } else {
          // D = 128, half CH: K rows own words tig*2 + CH; V rows own the half-words of parity CH
          if constexpr (!IS_V) {
            uint32_t* cw = reinterpret_cast<uint32_t*>(crow);
#pragma unroll
            for (int tg = 0; tg < 4; ++tg) cw[2 * tg + CH] = words[2 * tg + CH];
          } else {
            uint16_t* hw16 = reinterpret_cast<uint16_t*>(crow);
#pragma unroll
            for (int w = 0; w < 8; ++w)
              hw16[2 * w + CH] = static_cast<uint16_t>(CH ? (words[w] >> 16) : (words[w] & 0xFFFFu));
          }
#pragma unroll
          for (int gq = 0; gq < GPH; ++gq) szp[CH * GPH + gq] = szw[CH * GPH + gq];
        }
      };
      using I0 = std::integral_constant<int, 0>;
      using I1 = std::integral_constant<int, HALVES - 1>;
      using VT = std::integral_constant<bool, true>;
      using VF = std::integral_constant<bool, false>;
      if (ch == 0) {
        if (is_v) quant_store(I0{}, VT{}); else quant_store(I0{}, VF{});
      } else {
        if (is_v) quant_store(I1{}, VT{}); else quant_store(I1{}, VF{});
      }
      if (kind == 2 && ch == 0) {
        if (req < 0 || req >= g.max_req) {
          flag_error(a.status, kDevBadSlot);
        } else {
          const size_t sbase = ((size_t)a.layer * g.max_req + req) * g.slab_req_elems();
          const int slot = pos < g.S ? pos : g.S + (pos - g.S) % g.W;
          uint4* dst = reinterpret_cast<uint4*>(a.slab + sbase + (((size_t)h * 2 + (is_v ? 1 : 0)) * g.window() + slot) * D);
          const uint4* in = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(src) +
                                                           ((size_t)token * g.Hkv + h) * D);
#pragma unroll
          for (int q = 0; q < D / 8; ++q) dst[q] = in[q];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kEpiWarps) tmem_dealloc(tmem, L::TMEM_COLS);
}

PFN_cuTensorMapEncodeTiled_v12000 tc_get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D map over rows of D BF16 values (rows = tokens x kv heads), box 64 x 128, 128-byte swizzle.
int make_row_map(CUtensorMap* map, const void* base, long long rows, int D) {
  auto enc = tc_get_encode();
  if (!enc) return (int)cudaErrorNotSupported;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)kTileM};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : (int)cudaErrorInvalidValue;
}

// 3-D map over [tokens][Hkv][D] BF16, box 64 x 1 x 128: 128 tokens of one kv head (the same
// shared-memory image as a 64 x 128 box of the 2-D map).
int make_head_row_map(CUtensorMap* map, const void* base, long long tokens, int hkv, int D) {
  auto enc = tc_get_encode();
  if (!enc) return (int)cudaErrorNotSupported;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)hkv, (cuuint64_t)tokens};
  cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)hkv * D * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)kTileM};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : (int)cudaErrorInvalidValue;
}

// The row tensor maps of recent calls, keyed by (base, rows, kv heads, D, form): a map encodes
// only the address, sizes and strides, so one that matches is the map the call would build.
// Repeated writes from the same staging buffers (a layer loop) then skip the encode.
int cached_row_map(CUtensorMap* map, const void* base, long long rows, int hkv, int D, bool per_head) {
  struct Entry {
    const void* base;
    long long rows;
    int hkv, d, per_head;
    CUtensorMap map;
  };
  constexpr int kEntries = 16;
  static std::mutex mu;
  static Entry table[kEntries];
  static int used = 0, next = 0;
  {
    std::lock_guard<std::mutex> lk(mu);
    for (int i = 0; i < used; ++i) {
      const Entry& e = table[i];
      if (e.base == base && e.rows == rows && e.hkv == hkv && e.d == D && e.per_head == (int)per_head) {
        *map = e.map;
        return 0;
      }
    }
  }
  const int r = per_head ? make_head_row_map(map, base, rows, hkv, D) : make_row_map(map, base, rows, D);
  if (r) return r;
  std::lock_guard<std::mutex> lk(mu);
  Entry& e = table[next];
  e = Entry{base, rows, hkv, D, (int)per_head, *map};
  next = (next + 1) % kEntries;
  if (used < kEntries) ++used;
  return 0;
}

template <int D, bool HAD>
int launch_write_tc_t(const WriteArgs& a, cudaStream_t s, bool pdl) {
  using L = TcPlan<D, HAD>;
  const bool rph = a.g.rph != 0;
  const long long rows = rph ? (long long)a.total_tokens : (long long)a.total_tokens * a.g.Hkv;
  const long long tiles = (rows + kTileM - 1) / kTileM;
  CUtensorMap mk, mv;
  int e = cached_row_map(&mk, a.K, rph ? (long long)a.total_tokens : rows, a.g.Hkv, D, rph);
  if (e) return e;
  if ((e = cached_row_map(&mv, a.V, rph ? (long long)a.total_tokens : rows, a.g.Hkv, D, rph))) return e;
  // at least 120 KB of shared memory: one CTA per SM, so the TMEM allocation never waits
  const int smem = L::SMEM > 120 * 1024 ? L::SMEM : 120 * 1024;
  cudaError_t ce = ensure_smem_limit(write_tc_kernel<D, HAD>, smem);
  if (ce != cudaSuccess) return (int)ce;
  // x2 (K, V): one CTA per SM; with a rotation per kv head, the same number of CTAs for every head
  int ctas = (int)(tiles < 76 ? tiles : 76);
  if (rph) {
    const long long per_head = tiles < 76 / a.g.Hkv ? tiles : (76 / a.g.Hkv > 0 ? 76 / a.g.Hkv : 1);
    ctas = (int)(per_head * a.g.Hkv);
  }
  return launch_pdl(write_tc_kernel<D, HAD>, dim3(ctas, 2), dim3(tc_threads<D>()), (size_t)smem, s, pdl, mk, mv, a);
}

}  // namespace

bool write_tc_supported(const WriteArgs& a) {
  return a.dtype == kDtypeBF16 && (a.g.D == 128 || a.g.D == 64) &&
         (reinterpret_cast<uintptr_t>(a.K) & 15) == 0 && (reinterpret_cast<uintptr_t>(a.V) & 15) == 0;
}

int launch_write_tc(const WriteArgs& a, void* stream, bool pdl) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((long long)a.total_tokens * a.g.Hkv == 0) return 0;
  if (a.hadamard) return a.g.D == 128 ? launch_write_tc_t<128, true>(a, s, pdl) : launch_write_tc_t<64, true>(a, s, pdl);
  return a.g.D == 128 ? launch_write_tc_t<128, false>(a, s, pdl) : launch_write_tc_t<64, false>(a, s, pdl);
}

}  // namespace oscar
