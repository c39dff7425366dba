// Extend (chunked prefill) attention over the mixed INT2 / BF16 paged cache on the
// 5th-generation tensor cores (tcgen05 + TMEM).
//
// Source: OSCAR technical summary (gist.science), section 2.2 B -- the serving kernel
// unpacks, dequantises and inverse-rotates the INT2 history and computes attention over
// it, compatible with paged attention and prefix caching; section 3 -- prefix reuse kept
// with the INT2 cache.  Request b holds prefix_lens[b] cached tokens (history INT2 in the
// rotated basis, sink and recent tokens BF16) and brings a chunk of new tokens; query i
// of the chunk attends to every cached token and, causally, to chunk tokens 0..i, whose
// keys and values are the chunk's own BF16 inputs.
//
// One CTA owns 128 query rows (chunk tokens x the query heads of one kv head, row r =
// token i0 + r / gq, head r % gq) and walks 64-key tiles: first the INT2 history tiles,
// then the BF16 window tiles, then the chunk's own tiles.  Per tile:
//   S = Q K^T into TMEM (two buffers, so the next tile's scores are computed while the
//   softmax reads this tile's), softmax by the row's own thread, P back into TMEM over
//   the tile's own scores, O += P V into TMEM.  History tiles take both A operands from TMEM (the rotated query planes,
//   the weights), so the tensor core reads only the unpacked keys and values from shared
//   memory, and their softmax waits for the previous tile's PV only to rescale.
// History tiles run in the rotated basis with f16 operands, each dequantised value split
// about its group's centre, z + c s = (z + 1.5 s) + (c - 1.5) s, so that the two parts do
// not cancel in the float32 accumulators (a group straddling zero has z near -1.5 s):
//   K operand  = (code - 1.5) * s * 2^(k_K + pos - 10)  (exact: an 8-bit scale times
//                +-0.5 or +-1.5),
//   Q operand  = q' * 2^(e_r + 10 - pos), split into f16 hi + lo (22 bits),
//   centre term = one more MMA (K = 16): the q' group sums Q_g in three f16 terms times
//                the centres m = z + 1.5 s in two (hi, lo), the four (five for d = 64)
//                largest of the six cross products,
//   V operand  = (code - 1.5) * s_V * 2^(k_V + pos - 10), with the V centres (hi and lo
//   rows) appended as 16 more B rows, so that one MMA with N = D + 16 also accumulates
//   sum_j p_j m_j; the slot factor 2^(10 - pos) and the centres are applied in the epilogue,
//   P as f16 hi + lo (weights <= 2^14), the row sum l kept in float32.
// BF16 tiles run in the plain basis with BF16 operands: Q as received (the query is BF16),
// P as three BF16 terms (24 bits; the values are unbounded BF16), K and V exactly
// as stored.  Both kinds share one running softmax reference per row; the two
// output accumulators (rotated and plain) are rescaled together.  The epilogue forms
// out = O_plain / l + (y / l) R_V^T on the tensor cores, y the rotated accumulator put
// back to value scale.
//
// Roles: warps 0-3 (softmax; thread r owns row r = TMEM lane r), warps 4-7 (the next
// tile into a shared-memory operand stage: INT2 pages bulk-copied two tiles ahead and
// unpacked, BF16 rows copied and V transposed; or, in the unpacked-prefix form, one bulk
// copy of the tile's image that a pre-pass formed once per call for all the request's
// query tiles), warp 8 (TMEM allocation, MMA issue).  The roles meet only at mbarriers:
// kv_full (a stage filled), s_full (scores in TMEM), p_full (weights in place),
// pv_done and kv_empty (a tile's PV done, its stage free), so the scores of
// tile j are computed while the softmax works on tile j - 1.  Every wait is bounded by
// %globaltimer: a timeout flags the status word and the CTA drains and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>
#include <utility>

#include "common.cuh"
#include "oscar_internal.h"

namespace oscar {
namespace {

#include "tc_common.cuh"

constexpr int kXRows = 128;                  // query rows per CTA (TMEM lanes)
constexpr int kXKeys = 64;                   // keys per tile
constexpr int kXThreads = 9 * 32;            // softmax 0-3, unpack 4-7 (warp 4 also copies pages), MMA 8
constexpr float kXLog2e = 1.4426950408889634f;
constexpr float kXRescaleLog2 = 8.f;         // the reference moves when a score exceeds it by more
constexpr float kXRescaleLog2Bf16 = 24.f;    // the same on BF16 tiles, whose weights go in as BF16 terms
constexpr float kXWeightShift = 6.f;         // weights 2^(s - m), m = reference - shift: at most 2^14

enum TileKind { kTileInt2 = 0, kTileWindow = 1, kTileChunk = 2 };

template <typename F, size_t... I>
__device__ __forceinline__ void static_for_impl(F&& f, std::index_sequence<I...>) {
  (f(std::integral_constant<int, (int)I>{}), ...);
}
template <int N, typename F>
__device__ __forceinline__ void static_for(F&& f) {
  static_for_impl(f, std::make_index_sequence<N>{});
}

// Shared memory plan (bytes from a 1024-aligned base).  Every operand tile is K-major
// with the 128-byte swizzle, 1024-aligned.
template <int D>
struct XLayout {
  static constexpr int G = D / 32;
  static constexpr int NST = 3;    // operand stages: tile j unpacked into stage j % NST
  static constexpr int NRAW = 3;   // raw page buffers: tile j's pages requested NRAW - 1 tiles ahead
  static constexpr int Q_PLANE = kXRows * D * 2;
  static constexpr int QHI = 0;    // the BF16 query of the BF16 tiles (the rotated planes live in TMEM)
  static constexpr int KT = 0, KT_BYTES = kXKeys * D * 2;         // [64 keys][D]
  static constexpr int KZ = KT + KT_BYTES, KZ_BYTES = kXKeys * 128;  // [64 keys][64], 16 columns used
  static constexpr int VT = KZ + KZ_BYTES, VT_BYTES = D * kXKeys * 2;  // [D channels][64 keys]
  static constexpr int ZV = VT + VT_BYTES, ZV_BYTES = 16 * 128;   // [16 (groups, padded)][64 keys]
  static constexpr int STAGE = ZV + ZV_BYTES;
  static constexpr int ST0 = QHI + Q_PLANE;
  static constexpr int RAW_BYTES = kXKeys * 3 * D / 4;           // 64 INT2 tokens: codes and (scale, zero) of K, V
  static constexpr int RAW0 = ST0 + NST * STAGE;
  static constexpr int BAR = RAW0 + NRAW * RAW_BYTES;
  // s_full[2], pv_done, kv_full[NST], kv_empty[NST], p_full[2], raw_full[NRAW], epi_copy,
  // epi_mma; then the TMEM slot, the abort flag
  static constexpr int NBAR = 2 + 1 + 2 * NST + 2 + NRAW + 2;
  static constexpr int BYTES = BAR + NBAR * 8 + 16;
  static constexpr int SMEM = BYTES + 1024;
  // epilogue reuse (after the last MMA): R_V as f16 hi and lo planes (the B operand of y R_V^T,
  // K-major, 128-byte swizzle) from 0, then 1/l [128]
  static constexpr int RP = 0, RP_BYTES = 2 * D * D * 2;
  static constexpr int LINV = (RP_BYTES + 1023) / 1024 * 1024;
  // TMEM columns
  // the V centre accumulator (16 columns) directly follows the rotated one: one PV MMA with
  // N = D + 16 reads the Zv rows that follow the Vt rows in shared memory
  static constexpr uint32_t C_S = 0, C_OROT = 2 * kXKeys, C_OZ = C_OROT + D, C_OPLAIN = C_OZ + 32;
  static constexpr uint32_t C_END = C_OPLAIN + D;
  // While the INT2 tiles run, the plain output is not yet in use: its D columns hold the
  // rotated query planes (hi, then lo: D / 2 columns each, a pair of channels per column),
  // the A operand of the INT2 score MMAs; the group-sum operand (16 f16) follows C_END.
  // The first BF16 tile's PV overwrites the plain output (its first MMA does not accumulate).
  static constexpr uint32_t C_QHI = C_OPLAIN, C_QLO = C_OPLAIN + D / 2, C_QZ = C_END;
  // Weights go back into TMEM over their tile's scores (a pair of keys per column: hi in the
  // first 32 columns, lo in the next 32); a BF16 tile's third term (lo2) goes to C_P2 + 32 (j & 1),
  // columns of the group-sum operand, which only the INT2 tiles before it read.
  static constexpr uint32_t C_P2 = C_END;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(STAGE % 1024 == 0 && ST0 % 1024 == 0, "operand tiles 1024-aligned");
  static_assert(C_QZ + 8 <= TMEM_COLS && C_P2 + kXKeys <= TMEM_COLS, "TMEM plan");
  static_assert(ZV == VT + D * 128, "Zv rows follow the Vt rows");
  static_assert(LINV + kXRows * 4 <= RAW0, "the R_V planes and 1/l fit below the raw buffers");
  static_assert(RAW0 % 16 == 0 && RAW_BYTES % 16 == 0, "bulk copy destinations 16-byte aligned");
  static_assert(SMEM <= 232448, "shared memory per CTA");
};

// ------------------------------------------------------------------ query rotation
// q' = q R_K for every (chunk token, query head) row, float32, into the workspace, on the
// tensor cores: a CTA takes 128 rows (the BF16 query as received, K-major with the 128-byte
// swizzle) against R_K^T split exactly into three BF16 planes (R = R1 + R2 + R3, 3 x 8
// significant bits covering float32's 24), built in shared memory; 3 x D/16 MMAs (the small
// planes first) into one float32 TMEM accumulator, which thread t reads for row t.  The last
// CTA writes R_V as f16 hi and lo planes (row n = output channel n, K-major with the 128-byte
// swizzle: the B operand of the epilogue's y R_V^T).
template <int D>
struct QrPlan {
  static constexpr int PLANE = D * D * 2;        // one BF16 plane of R_K^T
  static constexpr int A_OFF = 3 * PLANE;        // 128 query rows, BF16
  static constexpr int BAR = A_OFF + 128 * D * 2;
  static constexpr int SMEM = BAR + 16 + 1024;   // slack for the 1024-byte alignment of the base
};

template <int D>
__global__ void __launch_bounds__(128, 1) extend_qrot_kernel(ExtendArgs a) {
  using Q = QrPlan<D>;
  extern __shared__ uint8_t xq_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(xq_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + Q::BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + Q::BAR + 8);
  const int t = threadIdx.x, warp = t >> 5;
  const Geom& g = a.g;
  const long long rows = (long long)a.total_tokens * g.Hq;
  float* qrot = reinterpret_cast<float*>(a.ws + a.qrot_off);
  // blockIdx.y: the kv head whose rotation the CTA applies (0 with one rotation per layer)
  const int kvh = blockIdx.y;
  if (blockIdx.x == gridDim.x - 1) {
    uint8_t* rp = a.ws + a.rvp_off + (size_t)kvh * (2 * D * D * 2);
    const float* rv = a.R_V + (size_t)kvh * g.rot_stride();
    for (int item = t; item < D * D / 8; item += 128) {   // 8 consecutive k of row n
      const int n = item / (D / 8), k0 = 8 * (item % (D / 8));
      const float4 x0 = __ldg(reinterpret_cast<const float4*>(rv + (size_t)n * D + k0));
      const float4 x1 = __ldg(reinterpret_cast<const float4*>(rv + (size_t)n * D + k0 + 4));
      const float v[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        hi[q] = pack_half2(v[2 * q], v[2 * q + 1]);
        const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hi[q]));
        lo[q] = pack_half2(v[2 * q] - hf.x, v[2 * q + 1] - hf.y);
      }
      *reinterpret_cast<uint4*>(rp + sw128_offset(n, k0, D)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<uint4*>(rp + D * D * 2 + sw128_offset(n, k0, D)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    return;
  }
  // global row of local row l: one rotation per layer, rows 128 x + l of [tokens][Hq]; one per
  // kv head, the 128 / gq tokens x gq query heads of kv head kvh starting at token (128 / gq) x
  const int gq = g.gq();
  auto row_of = [&](int l) -> long long {
    if (!g.rph) return (long long)blockIdx.x * 128 + l;
    const long long tok = (long long)blockIdx.x * (128 / gq) + l / gq;
    return tok < a.total_tokens ? tok * g.Hq + (long long)kvh * gq + l % gq : rows;
  };
  {
    // The attention reads q' only for requests with INT2 history tiles: a CTA whose rows all
    // belong to requests without history (every request of a prefill from scratch) stops here.
    const long long tok0 = g.rph ? (long long)blockIdx.x * (128 / gq) : (long long)blockIdx.x * 128 / g.Hq;
    long long tok1 = g.rph ? tok0 + 128 / gq - 1 : ((long long)blockIdx.x * 128 + 127) / g.Hq;
    if (tok1 >= a.total_tokens) tok1 = a.total_tokens - 1;
    auto request_of = [&](long long tk) {   // largest b with cu_seqlens[b] <= tk
      int lo = 0, hi = a.batch - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.cu_seqlens[mid] <= tk) lo = mid; else hi = mid - 1;
      }
      return lo;
    };
    if (tok0 <= tok1) {
      const int b0 = request_of(tok0), b1 = request_of(tok1);
      bool need = b1 - b0 > 64;
      for (int bb = b0; !need && bb <= b1; ++bb) need = a.prefix_lens[bb] - g.W > g.S;
      if (!need) return;
    }
  }
  // R_K^T as three BF16 planes (row n = column n of R_K); item = (n, k-octet)
  const float* R = a.R_K + (size_t)kvh * g.rot_stride();
  for (int item = t; item < D * D / 8; item += 128) {
    const int n = item % D, k0 = (item / D) * 8;
    uint32_t pk[3][4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t lo[3], hi[3];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float r = __ldg(R + (size_t)(k0 + 2 * q + e) * D + n);
        const __nv_bfloat16 p1 = __float2bfloat16_rn(r);
        const float r1 = r - __bfloat162float(p1);
        const __nv_bfloat16 p2 = __float2bfloat16_rn(r1);
        const __nv_bfloat16 p3 = __float2bfloat16_rn(r1 - __bfloat162float(p2));
        (e ? hi : lo)[0] = *reinterpret_cast<const uint16_t*>(&p1);
        (e ? hi : lo)[1] = *reinterpret_cast<const uint16_t*>(&p2);
        (e ? hi : lo)[2] = *reinterpret_cast<const uint16_t*>(&p3);
      }
#pragma unroll
      for (int p = 0; p < 3; ++p) pk[p][q] = lo[p] | (hi[p] << 16);
    }
    const uint32_t off = sw128_offset(n, k0, D);
#pragma unroll
    for (int p = 0; p < 3; ++p)
      *reinterpret_cast<uint4*>(sm + p * Q::PLANE + off) = make_uint4(pk[p][0], pk[p][1], pk[p][2], pk[p][3]);
  }
  // the query rows, BF16 as received (rows past the end zero)
  for (int idx = t; idx < 128 * D / 8; idx += 128) {
    const int l = idx / (D / 8), c8 = idx % (D / 8);
    const long long r = row_of(l);
    const uint4 v = r < rows ? *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) + (size_t)r * D + 8 * c8)
                             : make_uint4(0u, 0u, 0u, 0u);
    *reinterpret_cast<uint4*>(sm + Q::A_OFF + sw128_offset(l, 8 * c8, 128)) = v;
  }
  if (t == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(tslot, D);
  // the planes and rows were written by ordinary stores; the MMAs read them through the async proxy
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (t == 0) {
    const uint32_t idesc = idesc_bf16_f32(128, D);
    const uint32_t a_base = smem_u32(sm + Q::A_OFF), b_base = smem_u32(sm);
#pragma unroll
    for (int pp = 0; pp < 3; ++pp) {
      const int p = 2 - pp;   // the small planes first: each MMA rounds relative to the running sum
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t ak = (uint32_t)((kk >> 2) * 128 * 128 + (kk & 3) * 32);
        const uint32_t bk = (uint32_t)(p * Q::PLANE + (kk >> 2) * D * 128 + (kk & 3) * 32);
        tc_mma_bf16(tmem, smem_desc_sw128(a_base + ak), smem_desc_sw128(b_base + bk), idesc, (pp | kk) ? 1u : 0u);
      }
    }
    tc_commit(bar);
  }
  const bool ok = mbar_wait_bounded(bar, 0, a.status);
  tc_fence_after();
  // thread t reads row t (TMEM lane t)
  const long long r = row_of(t);
#pragma unroll 1
  for (int cb = 0; cb < D / 32; ++cb) {
    uint32_t v[32];
    tmem_ld32_nowait(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(32 * cb), v);
    tmem_wait_ld();
    if (ok && r < rows) {
      float4* dst = reinterpret_cast<float4*>(qrot + (size_t)r * D + 32 * cb);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]), __uint_as_float(v[4 * j + 2]),
                             __uint_as_float(v[4 * j + 3]));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, D);
}

// ------------------------------------------------------------------ attention
// named barrier 1 among the 128 unpack threads, returning whether any of them passed true
__device__ __forceinline__ bool unpack_bar_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\tbar.red.or.pred po, 1, 128, pi;\n\t"
      "selp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ uint32_t half2_bits(float lo_elem, float hi_elem) { return pack_half2(lo_elem, hi_elem); }
// 2^e for e in the float32 normal range
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((e + 127) << 23); }

// Bounded mbarrier wait for the role warps: the waiting thread is suspended in the barrier
// (try_wait with a suspend-time hint) rather than spinning, so it leaves the issue slots to
// the working warps; the limit is kWaitLimitNs as for every wait.
__device__ __forceinline__ bool xwait(uint64_t* bar, uint32_t parity, int* status) {
  return mbar_wait_sleep_bounded(bar, parity, status);
}

// f16 pair (1.5 * 2^(pos - 10), same): the centring constant of a code slot at bit pos
__host__ __device__ constexpr uint32_t centre_pair(int pos) {
  // f16 of 1.5 * 2^(pos - 10): exponent field pos - 10 + 15, mantissa 0x200
  return ((uint32_t)((pos + 5) << 10 | 0x200)) * 0x10001u;
}
// r = s * c * 2^(pos - 10) (from scale_codes with n2 = -s) -> s * (c - 1.5) * 2^(pos - 10),
// one f16 fused multiply-add per pair, exact (the result has at most 10 significant bits)
__device__ __forceinline__ uint32_t centre_codes(uint32_t r, uint32_t n2, uint32_t kc) {
  const __half2 rv = *reinterpret_cast<const __half2*>(&r);
  const __half2 nv = *reinterpret_cast<const __half2*>(&n2);
  const __half2 cv = *reinterpret_cast<const __half2*>(&kc);
  const __half2 o = __hfma2(nv, cv, rv);
  return *reinterpret_cast<const uint32_t*>(&o);
}
// group centre m = z + 1.5 s (from a (scale, zero) word) times 2^k as f16 hi + lo (exact)
__device__ __forceinline__ void centre_hi_lo(uint32_t w, uint32_t k23, __half& hi, __half& lo) {
  const float m = zero_times_pow2(w, k23) + 1.5f * scale_times_pow2(w, k23);
  hi = __float2half_rn(m);
  lo = __float2half_rn(m - __half2float(hi));
}
// centre-term columns: term t pairs query term centre_q_term(t) (0 hi, 1 lo, 2 lo2 of Q_g)
// with centre term centre_z_term(t) (0 hi, 1 lo of m); G groups per term, 16 columns in all
__host__ __device__ constexpr int centre_q_term(int t) { return t == 3 ? 2 : (t == 1 || t == 4 ? 1 : 0); }
__host__ __device__ constexpr int centre_z_term(int t) { return t == 2 || t == 4 ? 1 : 0; }
template <int G>
__host__ __device__ constexpr int kCentreTerms() { return 16 / G < 5 ? 16 / G : 5; }

// What one CTA walks: nR INT2 tiles (positions 64u, u >= u0), nW window tiles (slab
// slots 64w), nC chunk tiles (chunk keys 64c).
struct XTiles {
  int nR, nW, nC, u0;
  int S, hist_end, n_sink, n_rec;   // history [S, hist_end); window slots [0, n_sink) and [S, S + n_rec)
  __device__ int n() const { return nR + nW + nC; }
  __device__ int kind(int j) const { return j < nR ? kTileInt2 : (j < nR + nW ? kTileWindow : kTileChunk); }
  __device__ int base(int j) const {
    return j < nR ? 64 * (u0 + j) : (j < nR + nW ? 64 * (j - nR) : 64 * (j - nR - nW));
  }
};

// Unpacks one 64-key INT2 history tile (its pages contiguous at raw: block i holds keys
// [i P, (i + 1) P)) into the operand tiles of a stage (Kt, Kz, Vt, Zv at stg), by 128
// threads u = 0..127.  Keys outside the history [S, hist_end) get zero operands.  Used by the
// attention kernel on its own shared-memory stage and by the pre-pass that dequantises a
// prefix once per call.
template <int D>
__device__ __forceinline__ void unpack_int2_tile(const uint8_t* raw, uint8_t* stg, int u, int base, int S,
                                                 int hist_end, int pshift, int pmask, size_t BB, const Geom& g,
                                                 uint32_t magic, uint32_t kK23, uint32_t kV23) {
  using L = XLayout<D>;
  constexpr int G = L::G;
  // K codes -> code * s * 2^(k_K + pos - 10); thread (key, w) writes channels [64w, 64w + 64),
  // groups 2w and 2w + 1, and those groups' centres m = z + 1.5 s: Kz row key, column t G + g
  // holds term centre_z_term(t) of m (the query side matches it)
  if (u < kXKeys * (D / 64)) {
    const int key = u / (D / 64), w = u % (D / 64);
    const bool ok = (base + key >= S && base + key < hist_end);
    const uint8_t* kb = raw + (key >> pshift) * BB;
    const int slot = key & pmask;
    uint32_t wd[4], w6[4];
#pragma unroll
    for (int tg = 0; tg < 4; ++tg) {
      wd[tg] = *reinterpret_cast<const uint32_t*>(kb + slot * (D / 4) + (tg * (D / 64) + w) * 4);
      w6[tg] = wd[tg] >> 6;
    }
    uint32_t szw[G];
#pragma unroll
    for (int gg = 0; gg < G; ++gg)
      szw[gg] = *reinterpret_cast<const uint32_t*>(kb + g.k_sz_off() + slot * (D / 8) + gg * 4);
    const int gA = 2 * w;
    const uint32_t sA = szw[gA], sB = szw[gA + 1];
    const uint32_t nA = ok ? half2_bits(neg_scale_times_pow2(sA, kK23), neg_scale_times_pow2(sA, kK23)) : 0u;
    const uint32_t nB = ok ? half2_bits(neg_scale_times_pow2(sB, kK23), neg_scale_times_pow2(sB, kK23)) : 0u;
    static_for<8>([&](auto X) {
      constexpr int x = decltype(X)::value;
      const uint32_t n2 = x < 4 ? nA : nB;
      constexpr uint32_t kc = centre_pair(slot_pos(x));
      uint4 c;
      c.x = centre_codes(scale_codes(magic_slot<x>(wd[0], w6[0], magic), n2), n2, kc);
      c.y = centre_codes(scale_codes(magic_slot<x>(wd[1], w6[1], magic), n2), n2, kc);
      c.z = centre_codes(scale_codes(magic_slot<x>(wd[2], w6[2], magic), n2), n2, kc);
      c.w = centre_codes(scale_codes(magic_slot<x>(wd[3], w6[3], magic), n2), n2, kc);
      *reinterpret_cast<uint4*>(stg + L::KT + sw128_offset(key, 8 * (8 * w + x), kXKeys)) = c;
    });
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      __half mh, ml;
      centre_hi_lo(ok ? (e ? sB : sA) : 0u, kK23, mh, ml);
      const __half mt[2] = {mh, ml};
#pragma unroll
      for (int tt = 0; tt < kCentreTerms<G>(); ++tt)
        *reinterpret_cast<__half*>(stg + L::KZ + sw128_offset(key, tt * G + gA + e, kXKeys)) = mt[centre_z_term(tt)];
    }
  }
  // V codes -> code * s_V * 2^(k_V + pos - 10), transposed: thread (half-word hw, keys 8kb..8kb+7)
  if (u < (D / 8) * 8) {
    const int hw = u % (D / 8), kb8 = u / (D / 8);
    const int chbase = 64 * (hw % (D / 64)) + hw / (D / 64);
    const int gA = chbase / 32;
    uint32_t W[4], W6[4], nA[4], nB[4];

#pragma unroll
    for (int p = 0; p < 4; ++p) {
      uint32_t hv[2];
      float sa[2], sb[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int key = 8 * kb8 + 2 * p + e;
        const bool ok = (base + key >= S && base + key < hist_end);
        const uint8_t* vb = raw + (key >> pshift) * BB;
        const int slot = key & pmask;
        hv[e] = *reinterpret_cast<const uint16_t*>(vb + g.v_codes_off() + slot * (D / 4) + hw * 2);
        const uint32_t* szr = reinterpret_cast<const uint32_t*>(vb + g.v_sz_off() + slot * (D / 8));
        sa[e] = ok ? neg_scale_times_pow2(szr[gA], kV23) : 0.f;
        sb[e] = ok ? neg_scale_times_pow2(szr[gA + 1], kV23) : 0.f;
      }
      W[p] = hv[0] | (hv[1] << 16);
      W6[p] = W[p] >> 6;
      nA[p] = half2_bits(sa[0], sa[1]);
      nB[p] = half2_bits(sb[0], sb[1]);
    }
    static_for<8>([&](auto X) {
      constexpr int s = decltype(X)::value;
      constexpr uint32_t kc = centre_pair(slot_pos(s));
      uint4 c;
      c.x = centre_codes(scale_codes(magic_slot<s>(W[0], W6[0], magic), s < 4 ? nA[0] : nB[0]), s < 4 ? nA[0] : nB[0], kc);
      c.y = centre_codes(scale_codes(magic_slot<s>(W[1], W6[1], magic), s < 4 ? nA[1] : nB[1]), s < 4 ? nA[1] : nB[1], kc);
      c.z = centre_codes(scale_codes(magic_slot<s>(W[2], W6[2], magic), s < 4 ? nA[2] : nB[2]), s < 4 ? nA[2] : nB[2], kc);
      c.w = centre_codes(scale_codes(magic_slot<s>(W[3], W6[3], magic), s < 4 ? nA[3] : nB[3]), s < 4 ? nA[3] : nB[3], kc);
      *reinterpret_cast<uint4*>(stg + L::VT + sw128_offset(chbase + 8 * s, 8 * kb8, D)) = c;
    });
    // the centres of groups gA, gA + 1 for one key each of the 8 threads that share kb8 and
    // gA: Zv rows g (hi) and G + g (lo), column key
    const int ckey = 8 * kb8 + hw / (D / 64);
    const bool cok = (base + ckey >= S && base + ckey < hist_end);
    const uint32_t* cszr = reinterpret_cast<const uint32_t*>(raw + (ckey >> pshift) * BB + g.v_sz_off() +
                                                             (ckey & pmask) * (D / 8));
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      __half mh, ml;
      centre_hi_lo(cok ? cszr[gA + e] : 0u, kV23, mh, ml);
      *reinterpret_cast<__half*>(stg + L::ZV + sw128_offset(gA + e, ckey, 16)) = mh;
      *reinterpret_cast<__half*>(stg + L::ZV + sw128_offset(G + gA + e, ckey, 16)) = ml;
    }
  }
}

// Where the K / V rows of a BF16 tile come from: window tiles read the request's slab slots
// (sink slots [0, n_sink), recent slots [S, S + n_rec)), chunk tiles the call's own K / V rows
// (chunk keys below kend); other keys are zero.
struct PlainSrc {
  int kind, base;
  int n_sink, S, n_rec, kend, c0, kvh, Hkv, window, D;
  const uint16_t* slab_req;   // this request's and kv head's K slab (V follows after window rows)
  const uint16_t* K_new;
  const uint16_t* V_new;
  __device__ const uint16_t* row(int key, int kv) const {
    if (kind == kTileWindow) {
      const int slot = base + key;
      const bool ok = slot < n_sink || (slot >= S && slot < S + n_rec);
      return ok ? slab_req + ((size_t)kv * window + slot) * D : nullptr;
    }
    const int kc = base + key;
    if (kc >= kend) return nullptr;
    return (kv ? V_new : K_new) + ((size_t)(c0 + kc) * Hkv + kvh) * D;
  }
};

// BF16 window or chunk tile into a stage: K rows copied into the swizzled K tile, V rows
// transposed, by 128 threads u = 0..127.  Used by the attention kernel and by the pre-pass.
template <int D>
__device__ __forceinline__ void unpack_plain_tile(const PlainSrc& src, uint8_t* stg, int u) {
  using L = XLayout<D>;
  constexpr int KI = kXKeys * (D / 8) / 128;   // 16-byte K pieces per thread
  uint4 kv[KI];
#pragma unroll
  for (int m = 0; m < KI; ++m) {
    const int item = u + 128 * m;
    const int key = item / (D / 8), cc = item % (D / 8);
    const uint16_t* row = src.row(key, 0);
    kv[m] = row ? *reinterpret_cast<const uint4*>(row + 8 * cc) : make_uint4(0u, 0u, 0u, 0u);
  }
  uint4 vr[8];
  const bool vt = u < D;   // thread (channel block hw8, keys 8kb..8kb+7)
  const int hw8 = u % (D / 8), kb8 = u / (D / 8);
  if (vt) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint16_t* row = src.row(8 * kb8 + k, 1);
      vr[k] = row ? *reinterpret_cast<const uint4*>(row + 8 * hw8) : make_uint4(0u, 0u, 0u, 0u);
    }
  }
#pragma unroll
  for (int m = 0; m < KI; ++m) {
    const int item = u + 128 * m;
    const int key = item / (D / 8), cc = item % (D / 8);
    *reinterpret_cast<uint4*>(stg + L::KT + sw128_offset(key, 8 * cc, kXKeys)) = kv[m];
  }
  if (vt) {
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const uint32_t sel = (e & 1) ? 0x7632u : 0x5410u;
      uint32_t c[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const uint4 x = vr[2 * p], y = vr[2 * p + 1];
        const uint32_t xs = (e >> 1) == 0 ? x.x : ((e >> 1) == 1 ? x.y : ((e >> 1) == 2 ? x.z : x.w));
        const uint32_t ys = (e >> 1) == 0 ? y.x : ((e >> 1) == 1 ? y.y : ((e >> 1) == 2 ? y.z : y.w));
        c[p] = prmt(xs, ys, sel);
      }
      *reinterpret_cast<uint4*>(stg + L::VT + sw128_offset(8 * hw8 + e, 8 * kb8, D)) =
          make_uint4(c[0], c[1], c[2], c[3]);
    }
  }
}

// Pre-pass of the unpacked-prefix form: every tile that the attention CTAs of a request share
// (its INT2 history tiles, dequantised; its BF16 window tiles; its chunk's own tiles, the V rows
// transposed) is formed once per call into the workspace, as the image of an attention stage
// (XLayout<D>::STAGE bytes, padding zero), so that the CTAs of all the request's query tiles
// bulk-copy it instead of each forming it.  Per (request, kv head): prep_tiles INT2 tiles, then
// prep_wt window tiles, then prep_ct chunk tiles.  Grid (tile, kv head, request), 128 threads;
// tiles past a request's own exit at once.  A page outside the block table or the pool is
// flagged as in the attention kernel.
template <int D>
__global__ void __launch_bounds__(128) extend_unpack_kernel(ExtendArgs a) {
  using L = XLayout<D>;
  extern __shared__ __align__(1024) uint8_t xu_smem_raw[];
  uint8_t* stg = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(xu_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* raw = stg + L::STAGE;   // the tile's pages, contiguous
  const Geom& g = a.g;
  const int j = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int u = threadIdx.x;
  const int n_pre = a.prefix_lens[b];
  if (n_pre < 0 || (long long)n_pre > (long long)g.max_pages_per_req * g.P) return;   // flagged by the attention
  const int hist_end = max(g.S, n_pre - g.W);
  uint4* out = reinterpret_cast<uint4*>(
      a.prep + (((size_t)b * g.Hkv + kvh) * (a.prep_tiles + a.prep_wt + a.prep_ct) + j) * L::STAGE);
  if (j >= a.prep_tiles) {
    // a BF16 tile: window slots of the request's slab, or the chunk's own K / V rows
    PlainSrc ps;
    const int c0 = a.cu_seqlens[b], len = a.cu_seqlens[b + 1] - c0;
    ps.n_sink = min(g.S, n_pre);
    ps.S = g.S;
    ps.n_rec = n_pre > g.S ? n_pre - hist_end : 0;
    ps.kend = len;
    ps.c0 = c0;
    ps.kvh = kvh;
    ps.Hkv = g.Hkv;
    ps.window = g.window();
    ps.D = D;
    ps.K_new = a.K_new;
    ps.V_new = a.V_new;
    ps.slab_req = nullptr;
    if (j < a.prep_tiles + a.prep_wt) {
      const int w = j - a.prep_tiles;
      const int win_end = ps.n_rec > 0 ? g.S + ps.n_rec : ps.n_sink;
      if (64 * w >= win_end) return;
      const int req = a.req_slot[b];
      if (req < 0 || req >= g.max_req) return;   // flagged by the attention
      ps.kind = kTileWindow;
      ps.base = 64 * w;
      ps.slab_req = a.slab + ((size_t)a.layer * g.max_req + req) * g.slab_req_elems() + (size_t)kvh * 2 * g.window() * D;
    } else {
      const int c = j - a.prep_tiles - a.prep_wt;
      if (len < 0 || c0 < 0 || c0 + len > a.total_tokens || 64 * c >= len) return;   // flagged by the attention
      ps.kind = kTileChunk;
      ps.base = 64 * c;
    }
    for (int q = u; q < L::STAGE / 16; q += 128) reinterpret_cast<uint4*>(stg)[q] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    unpack_plain_tile<D>(ps, stg, u);
    __syncthreads();
    for (int q = u; q < L::STAGE / 16; q += 128) out[q] = reinterpret_cast<const uint4*>(stg)[q];
    return;
  }
  if (hist_end <= g.S) return;
  const int u0 = g.S / 64;
  if (j > (hist_end - 1) / 64 - u0) return;
  const int base = 64 * (u0 + j);
  const int pshift = __ffs(g.P) - 1, pmask = g.P - 1, nblk = kXKeys >> pshift;
  const size_t BB = g.block_bytes();
  const uint8_t* pool_l = a.pool + (size_t)a.layer * g.layer_pool_bytes();
  for (int bi = 0; bi < nblk; ++bi) {
    const int lp = (base >> pshift) + bi;
    const int p0 = lp << pshift;
    if (p0 + g.P <= g.S || p0 >= hist_end) continue;   // no history token in this page
    const int page = (lp < a.bt_stride && lp < g.max_pages_per_req) ? a.block_table[(size_t)b * a.bt_stride + lp] : -1;
    if (page < 0 || page >= g.num_pages) {
      if (u == 0) flag_error(a.status, kDevBadPage);
      continue;
    }
    const uint4* src = reinterpret_cast<const uint4*>(pool_l + ((size_t)page * g.Hkv + kvh) * BB);
    uint4* dst = reinterpret_cast<uint4*>(raw + bi * BB);
    for (int q = u; q < (int)(BB / 16); q += 128) dst[q] = src[q];
  }
  for (int q = u; q < L::STAGE / 16; q += 128) reinterpret_cast<uint4*>(stg)[q] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();
  unpack_int2_tile<D>(raw, stg, u, base, g.S, hist_end, pshift, pmask, BB, g, a.code_magic,
                      static_cast<uint32_t>(a.k_exp_K) << 23, static_cast<uint32_t>(a.k_exp_V) << 23);
  __syncthreads();
  for (int q = u; q < L::STAGE / 16; q += 128) out[q] = reinterpret_cast<const uint4*>(stg)[q];
}

// PREP: launched with the unpacked-prefix workspace (a second instantiation, so that the form
// without it compiles to the kernel that has no copy path at all)
template <int D, bool PREP>
__global__ void __launch_bounds__(kXThreads, 1) extend_attn_kernel(ExtendArgs a) {
  using L = XLayout<D>;
  constexpr int G = L::G;
  extern __shared__ __align__(1024) uint8_t x_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(x_smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* s_full = reinterpret_cast<uint64_t*>(smem + L::BAR);   // [2] scores of tile j in TMEM (commit)
  uint64_t* pv_done = s_full + 2;          // PV of tile j done (commit)
  uint64_t* kv_full = s_full + 3;          // [NST] stage j % NST holds tile j (one arrival per unpack warp)
  uint64_t* kv_empty = kv_full + L::NST;   // [NST] stage free again (commit after the tile's PV)
  // [2] weights of tile j in place (one arrival per softmax warp), one barrier per tile parity: the
  // softmax may finish tile j + 1 before the MMA thread has seen tile j's, never tile j + 2
  // (its scores need tile j's PV issued first)
  uint64_t* p_full = kv_empty + L::NST;
  uint64_t* raw_full = p_full + 2;         // [NRAW] raw buffer j % NRAW holds INT2 tile j's pages (bulk copies)
  uint64_t* epi_copy = raw_full + L::NRAW;  // epilogue: the R_V planes arrived
  uint64_t* epi_mma = epi_copy + 1;          // epilogue: y R_V^T done (commit)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::BAR + 8 * L::NBAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::BAR + 8 * L::NBAR + 4);

  const Geom& g = a.g;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.z, kvh = blockIdx.y;
  const int gq = g.gq();
  const int tq = kXRows / gq;                 // chunk tokens per CTA
  const int i0 = blockIdx.x * tq;
  const int c0 = a.cu_seqlens[b];
  const int len = a.cu_seqlens[b + 1] - c0;
  // the host sizes (max_chunk, total_tokens) must cover the device lengths: a chunk longer than
  // the grid or past the rotated rows would go partly uncomputed
  if (len < 0 || c0 < 0 || c0 + len > a.total_tokens || len > (int)gridDim.x * tq) {
    if (blockIdx.x == 0 && threadIdx.x == 0) flag_error(a.status, kDevBadLen);
    return;
  }
  if (i0 >= len) return;
  const int n_pre = a.prefix_lens[b];
  if (n_pre < 0 || (long long)n_pre > (long long)g.max_pages_per_req * g.P) {
    if (tid == 0) flag_error(a.status, kDevBadLen);
    return;
  }
  XTiles tl;
  tl.S = g.S;
  tl.hist_end = max(g.S, n_pre - g.W);
  tl.n_sink = min(g.S, n_pre);
  tl.n_rec = n_pre > g.S ? n_pre - max(g.S, n_pre - g.W) : 0;
  if (tl.hist_end > g.S) {
    tl.u0 = g.S / 64;
    tl.nR = (tl.hist_end - 1) / 64 - tl.u0 + 1;
  } else {
    tl.u0 = 0;
    tl.nR = 0;
  }
  const int win_end = tl.n_rec > 0 ? g.S + tl.n_rec : tl.n_sink;
  tl.nW = (win_end + 63) / 64;
  const int kend = min(len, i0 + tq);
  tl.nC = (kend + 63) / 64;
  const int n_tiles = tl.n();
  // unpacked-prefix form: this request's tiles were formed by the pre-pass
  const bool use_prep = PREP && a.prep != nullptr && tl.nR <= a.prep_tiles && tl.nW <= a.prep_wt && tl.nC <= a.prep_ct;
  int req = 0;
  if (tl.nW > 0) {
    req = a.req_slot[b];
    if (req < 0 || req >= g.max_req) {
      if (tid == 0) flag_error(a.status, kDevBadSlot);
      return;
    }
  }

  const uint32_t kK23 = static_cast<uint32_t>(a.k_exp_K) << 23;
  const uint32_t kV23 = static_cast<uint32_t>(a.k_exp_V) << 23;
  const uint8_t* pool_l = a.pool + (size_t)a.layer * g.layer_pool_bytes();
  const size_t BB = g.block_bytes();
  const uint16_t* slab_req =
      a.slab + ((size_t)a.layer * g.max_req + req) * g.slab_req_elems() + (size_t)kvh * 2 * g.window() * D;

  // ---------------- setup: barriers, TMEM, Zv padding rows
  if (warp == 8) {
    if (lane == 0) {
      mbar_init(&s_full[0], 1);
      mbar_init(&s_full[1], 1);
      mbar_init(pv_done, 1);
      for (int st = 0; st < L::NST; ++st) {
        mbar_init(&kv_full[st], 4);
        mbar_init(&kv_empty[st], 1);
      }
      mbar_init(&p_full[0], 4);
      mbar_init(&p_full[1], 4);
      for (int rb = 0; rb < L::NRAW; ++rb) mbar_init(&raw_full[rb], 1);
      mbar_init(epi_copy, 1);
      mbar_init(epi_mma, 1);
      *abort_flag = 0;
      fence_barrier_init();
    }
    __syncwarp();
    tmem_alloc(tmem_slot, L::TMEM_COLS);
  }
  // columns past the centre terms of every stage's Kz tile stay zero (the query side's
  // matching columns are zero too; a zero times a zero keeps the padding out of the scores)
  constexpr int PADC = 16 - kCentreTerms<G>() * G;
  if constexpr (PADC > 0) {
    for (int idx = tid; idx < L::NST * kXKeys * PADC; idx += kXThreads) {
      const int st = idx / (kXKeys * PADC), rem = idx % (kXKeys * PADC);
      const int key = rem / PADC, col = kCentreTerms<G>() * G + rem % PADC;
      *reinterpret_cast<__half*>(smem + L::ST0 + st * L::STAGE + L::KZ + sw128_offset(key, col, kXKeys)) =
          __float2half_rn(0.f);
    }
  }
  // rows 2G..15 of every stage's Zv tile stay zero (padding of the V centre term)
  for (int idx = tid; idx < L::NST * (16 - 2 * G) * 8; idx += kXThreads) {
    const int st = idx / ((16 - 2 * G) * 8), rem = idx % ((16 - 2 * G) * 8);
    const int row = 2 * G + rem / 8, ck = rem % 8;
    *reinterpret_cast<uint4*>(smem + L::ST0 + st * L::STAGE + L::ZV + sw128_offset(row, 8 * ck, 16)) =
        make_uint4(0u, 0u, 0u, 0u);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // ---------------- per-row state of the softmax threads (warps 0-3: row r = tid)
  const int r = tid & (kXRows - 1);
  const int qi = i0 + r / gq;
  const bool row_ok = qi < len;
  const size_t qrow = (size_t)(c0 + (row_ok ? qi : i0)) * g.Hq + (size_t)kvh * gq + r % gq;
  const float sm_log2 = kXLog2e * rsqrtf((float)D);
  float F_rot = 0.f;
  const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);

  // Q planes for INT2 tiles: q' * 2^(e + 10 - pos) as f16 hi + lo, and the group sums
  // Q_g * 2^e as three f16 terms; |q'| * 2^e < 32 keeps every operand below 2^15.  They
  // go to this row's TMEM lane (column c of a plane: channels 2c, 2c + 1), the A operand
  // of the INT2 score MMAs.
  auto write_q_rot = [&]() {
    const float4* src = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(a.ws + a.qrot_off) + qrow * D);
    float mx = 0.f, qg[G];
#pragma unroll
    for (int gg = 0; gg < G; ++gg) qg[gg] = 0.f;
    if (row_ok) {
#pragma unroll 8
      for (int c = 0; c < D / 4; ++c) {
        const float4 v = src[c];
        mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        qg[c / 8] += (v.x + v.y) + (v.z + v.w);
      }
    }
    int e = 0;
    if (mx > 0.f) {
      int E;
      frexpf(mx, &E);
      e = 5 - E;
    }
    F_rot = ldexpf(sm_log2, -e - a.k_exp_K);
#pragma unroll 1
    for (int mg = 0; mg < D / 32; ++mg) {   // 16 columns (32 channels) per store
      uint32_t hi[16], lo[16];
#pragma unroll
      for (int mi = 0; mi < 4; ++mi) {
        const int m = 4 * mg + mi;   // channels 8m .. 8m + 7: columns 4m .. 4m + 3
        const float f = ldexpf(1.f, e + 10 - slot_pos(m & 7));
        float v[8];
        if (row_ok) {
          const float4 x0 = src[2 * m], x1 = src[2 * m + 1];
          v[0] = x0.x; v[1] = x0.y; v[2] = x0.z; v[3] = x0.w; v[4] = x1.x; v[5] = x1.y; v[6] = x1.z; v[7] = x1.w;
        } else {
#pragma unroll
          for (int k = 0; k < 8; ++k) v[k] = 0.f;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float x0 = v[2 * k] * f, x1 = v[2 * k + 1] * f;
          hi[4 * mi + k] = half2_bits(x0, x1);
          const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hi[4 * mi + k]));
          lo[4 * mi + k] = half2_bits(x0 - hf.x, x1 - hf.y);
        }
      }
      tmem_st16(lane_base + L::C_QHI + (uint32_t)(16 * mg), hi);
      tmem_st16(lane_base + L::C_QLO + (uint32_t)(16 * mg), lo);
    }
    __half hz[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) hz[k] = __float2half_rn(0.f);
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
      const float x = ldexpf(qg[gg], e);
      const __half h1 = __float2half_rn(x);
      const float r1 = x - __half2float(h1);
      const __half h2 = __float2half_rn(r1);
      const __half h3 = __float2half_rn(r1 - __half2float(h2));
      const __half qt[3] = {h1, h2, h3};
#pragma unroll
      for (int tt = 0; tt < kCentreTerms<G>(); ++tt) hz[tt * G + gg] = qt[centre_q_term(tt)];
    }
    uint32_t hz2[8];
#pragma unroll
    for (int c = 0; c < 8; ++c)
      hz2[c] = static_cast<uint32_t>(__half_as_ushort(hz[2 * c])) |
               (static_cast<uint32_t>(__half_as_ushort(hz[2 * c + 1])) << 16);
    tmem_st8(lane_base + L::C_QZ, hz2);
  };
  // Q plane for BF16 tiles, in shared memory: the BF16 query itself (exact in one plane)
  auto write_q_plain = [&]() {
#pragma unroll 4
    for (int m = 0; m < D / 8; ++m) {
      const uint4 w = row_ok ? *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.q) + qrow * D + 8 * m)
                             : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(smem + L::QHI + sw128_offset(r, 8 * m, kXRows)) = w;
    }
  };

  // ---------------- unpack threads (warps 4-7: u = tid - 128)
  const int u = tid - 128;
  auto hist_ok = [&](int t) { return t >= tl.S && t < tl.hist_end; };
  // INT2 pages of tile j into raw buffer j & 1 (one cp.async group per call, possibly empty)
  // page sizes are powers of two (16, 32, 64): block and slot of a key by shift and mask
  const int pshift = __ffs(g.P) - 1, pmask = g.P - 1, nblk = kXKeys >> pshift;
  constexpr int kMaxBlk = kXKeys / 16;
  // Page ids for the copying warp (warp 4): lane l holds the id of logical page 32 w + l of the
  // request's block table for the current 32-page window w (pid_cur) and for the next one
  // (pid_nxt, loaded a window ahead, so that its latency stays off the copy path).  -1: the
  // page holds no history token; -2: outside the block table.
  auto page_id_at = [&](int lp) -> int {
    const int p0 = lp << pshift;
    if (p0 + g.P <= tl.S || p0 >= tl.hist_end) return -1;
    return (lp < a.bt_stride && lp < g.max_pages_per_req) ? a.block_table[(size_t)b * a.bt_stride + lp] : -2;
  };
  int pid_cur = -1, pid_nxt = -1, win_cur = -2;
  // (copying warp, every lane) the page ids of INT2 tile j's blocks: nblk consecutive pages
  // from lp0, a multiple of nblk, so inside one window
  auto tile_pages = [&](int j, int (&pg)[kMaxBlk]) {
    const int lp0 = tl.base(j) >> pshift;
    const int w = lp0 >> 5;
    if (w != win_cur) {
      pid_cur = w == win_cur + 1 ? pid_nxt : page_id_at(32 * w + lane);
      pid_nxt = page_id_at(32 * (w + 1) + lane);
      win_cur = w;
    }
#pragma unroll
    for (int bi = 0; bi < kMaxBlk; ++bi) pg[bi] = __shfl_sync(0xffffffffu, pid_cur, (lp0 + bi) & 31);
  };
  // INT2 pages of tile j into raw buffer j % NRAW: one bulk copy per page block, issued by
  // lane 0 of the copying warp, completing on raw_full[j % NRAW] (an empty arrival when no
  // block is valid).  Every unpack thread has left the buffer's previous tile behind: the
  // caller passed the unpack barrier after that tile.
  auto issue_raw = [&](int j, const int (&pg)[kMaxBlk]) {
    if (j >= tl.nR) return;
    uint8_t* dst0 = smem + L::RAW0 + (j % L::NRAW) * L::RAW_BYTES;
    uint64_t* bar = &raw_full[j % L::NRAW];
    uint32_t bytes = 0;
#pragma unroll
    for (int bi = 0; bi < kMaxBlk; ++bi) {
      const int page = pg[bi];
      if (bi >= nblk || page == -1) continue;
      if (page < 0 || page >= g.num_pages) {
        flag_error(a.status, kDevBadPage);
        continue;
      }
      bytes += (uint32_t)BB;
    }
    mbar_arrive_expect_tx(bar, bytes);
#pragma unroll
    for (int bi = 0; bi < kMaxBlk; ++bi) {
      const int page = pg[bi];
      if (bi >= nblk || page < 0 || page >= g.num_pages) continue;
      bulk_g2s(dst0 + bi * BB, pool_l + ((size_t)page * g.Hkv + kvh) * BB, (uint32_t)BB, bar);
    }
  };
  auto unpack_int2 = [&](int j, uint8_t* stg) {
    unpack_int2_tile<D>(smem + L::RAW0 + (j % L::NRAW) * L::RAW_BYTES, stg, u, tl.base(j), tl.S, tl.hist_end,
                        pshift, pmask, BB, g, a.code_magic, kK23, kV23);
  };
  auto plain_src = [&](int j) {
    PlainSrc ps;
    ps.kind = tl.kind(j);
    ps.base = tl.base(j);
    ps.n_sink = tl.n_sink;
    ps.S = tl.S;
    ps.n_rec = tl.n_rec;
    ps.kend = kend;
    ps.c0 = c0;
    ps.kvh = kvh;
    ps.Hkv = g.Hkv;
    ps.window = g.window();
    ps.D = D;
    ps.slab_req = slab_req;
    ps.K_new = a.K_new;
    ps.V_new = a.V_new;
    return ps;
  };
  auto unpack_plain = [&](int j, uint8_t* stg) { unpack_plain_tile<D>(plain_src(j), stg, u); };
  // tile j into stage j % NST; false when an INT2 tile's pages did not arrive in time (the
  // status word is flagged; the caller stops at its next barrier)
  auto unpack = [&](int j) -> bool {
    uint8_t* stg = smem + L::ST0 + (j % L::NST) * L::STAGE;
    if (tl.kind(j) != kTileInt2) {
      unpack_plain(j, stg);
      return true;
    }
    if (!__all_sync(0xffffffffu, xwait(&raw_full[j % L::NRAW], (uint32_t)((j / L::NRAW) & 1), a.status)))
      return false;
    unpack_int2(j, stg);
    return true;
  };

  // ---------------- MMA issue (warp 8, lane 0)
  const uint32_t sbase = smem_u32(smem);
  // descriptors: the start-address field is (address >> 4) in the low 14 bits, so an
  // offset inside a tile is added to a base descriptor directly
  const uint64_t dQHI = smem_desc_sw128(sbase + L::QHI);
  const uint64_t dST = smem_desc_sw128(sbase + L::ST0);
  auto dadd = [](uint64_t d, uint32_t off) { return d + (uint64_t)(off >> 4); };
  auto issue_qk = [&](int j) {
    const uint32_t soff = (uint32_t)((j % L::NST) * L::STAGE);
    const uint32_t dS = tmem + L::C_S + (uint32_t)((j & 1) * kXKeys);
    if (tl.kind(j) == kTileInt2) {
      // A = the rotated query planes in TMEM (8 columns per K = 16 step), B = the key tile
      const uint32_t idesc = idesc_f16_f32(kXRows, kXKeys);
#pragma unroll
      for (int pl = 0; pl < 2; ++pl)
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t bk = (uint32_t)((kk >> 2) * kXKeys * 128 + (kk & 3) * 32);
          tc_mma_ts(dS, tmem + (pl ? L::C_QLO : L::C_QHI) + (uint32_t)(8 * kk), dadd(dST, soff + L::KT + bk), idesc,
                    (pl | kk) ? 1u : 0u);
        }
      tc_mma_ts(dS, tmem + L::C_QZ, dadd(dST, soff + L::KZ), idesc, 1u);
    } else {
      // the BF16 query, exact in one plane, from shared memory
      const uint32_t idesc = idesc_bf16_f32(kXRows, kXKeys);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t ak = (uint32_t)((kk >> 2) * kXRows * 128 + (kk & 3) * 32);
        const uint32_t bk = (uint32_t)((kk >> 2) * kXKeys * 128 + (kk & 3) * 32);
        tc_mma(dS, dadd(dQHI, ak), dadd(dST, soff + L::KT + bk), idesc, kk ? 1u : 0u);
      }
    }
  };
  auto issue_pv = [&](int j) {
    const uint32_t soff = (uint32_t)((j % L::NST) * L::STAGE);
    if (tl.kind(j) == kTileInt2) {
      // A = the weights, written by the softmax over this tile's scores in TMEM (hi in the
      // first 32 columns, lo in the next 32; a pair of keys per column)
      const uint32_t pcol = tmem + L::C_S + (uint32_t)((j & 1) * kXKeys);
#pragma unroll
      for (int pl = 0; pl < 2; ++pl)
#pragma unroll
        for (int kk = 0; kk < kXKeys / 16; ++kk)
          tc_mma_ts(tmem + L::C_OROT, pcol + (uint32_t)(32 * pl + 8 * kk), dadd(dST, soff + L::VT + kk * 32),
                    idesc_f16_f32(kXRows, D + 16), 1u);
    } else {
      // P as three BF16 terms (24 bits): window and chunk values are unbounded BF16.  The
      // first BF16 tile starts the plain accumulator, whose columns held the query planes.
      const uint32_t pcol = tmem + L::C_S + (uint32_t)((j & 1) * kXKeys);
      const uint32_t p2col = tmem + L::C_P2 + (uint32_t)((j & 1) * (kXKeys / 2));
#pragma unroll
      for (int pl = 0; pl < 3; ++pl)
#pragma unroll
        for (int kk = 0; kk < kXKeys / 16; ++kk)
          tc_mma_ts(tmem + L::C_OPLAIN, (pl < 2 ? pcol + (uint32_t)(32 * pl) : p2col) + (uint32_t)(8 * kk),
                    dadd(dST, soff + L::VT + kk * 32), idesc_bf16_f32(kXRows, D),
                    (j == tl.nR && pl == 0 && kk == 0) ? 0u : 1u);
    }
  };

  // ---------------- softmax of tile i (warps 0-3); false on a wait timeout
  float m_ref = -INFINITY, l_run = 0.f;
  bool ref_set = false;   // the reference has been placed by a visible key
  auto softmax_tile = [&](int i) -> bool {
    const int kind = tl.kind(i), base = tl.base(i);
    // waits are made warp-uniform: the TMEM accesses below are warp-collective.  With the tiles
    // copied (PREP) no unpack work shares the schedulers, and spinning on the scores reacts
    // sooner than suspending in the barrier (4 x (32K + 2K): 10.78 -> 10.63 ms)
    const bool s_ok = PREP ? mbar_wait_bounded(&s_full[i & 1], (uint32_t)(i >> 1) & 1, a.status)
                           : xwait(&s_full[i & 1], (uint32_t)(i >> 1) & 1, a.status);
    if (!__all_sync(0xffffffffu, s_ok)) return false;
    tc_fence_after();
    uint32_t s0[32], s1[32];
    tmem_ld32_nowait(lane_base + L::C_S + (uint32_t)((i & 1) * kXKeys), s0);
    tmem_ld32_nowait(lane_base + L::C_S + (uint32_t)((i & 1) * kXKeys + 32), s1);
    tmem_wait_ld();
    int a0 = 0, a1 = 0, b0 = 0, b1 = 0;   // visible keys [a0, a1) U [b0, b1)
    if (kind == kTileInt2) {
      a0 = max(0, tl.S - base);
      a1 = min(kXKeys, tl.hist_end - base);
    } else if (kind == kTileWindow) {
      a1 = min(kXKeys, tl.n_sink - base);
      b0 = max(0, tl.S - base);
      b1 = min(kXKeys, tl.S + tl.n_rec - base);
    } else {
      a1 = min(kXKeys, qi - base + 1);
    }
    const float F = kind == kTileInt2 ? F_rot : sm_log2;   // > 0: the maximum can be taken on raw values
    float sc[kXKeys];   // raw accumulator values, invisible keys at -inf
    float mraw = -INFINITY;
    if (a0 <= 0 && a1 >= kXKeys) {
#pragma unroll
      for (int jj = 0; jj < kXKeys; ++jj) {
        sc[jj] = __uint_as_float(jj < 32 ? s0[jj] : s1[jj - 32]);
        mraw = fmaxf(mraw, sc[jj]);
      }
    } else {
#pragma unroll
      for (int jj = 0; jj < kXKeys; ++jj) {
        const bool vis = (jj >= a0 && jj < a1) || (jj >= b0 && jj < b1);
        sc[jj] = vis ? __uint_as_float(jj < 32 ? s0[jj] : s1[jj - 32]) : -INFINITY;
        mraw = fmaxf(mraw, sc[jj]);
      }
    }
    const float mloc = mraw * F;
    float alpha = 1.f;
    // Weights 2^(score - m_ref) stay below 2^(shift + rescale): 2^14 on INT2 tiles (f16 operands);
    // on BF16 tiles (BF16 terms, float32 sums) the reference may lag by 24 before it moves, which
    // spares the rescale of both accumulators on most tiles of a growing causal chunk
    const float thr =
        ref_set ? m_ref + kXWeightShift + (kind == kTileInt2 ? kXRescaleLog2 : kXRescaleLog2Bf16) : -INFINITY;
    if (mloc > thr) {
      const float nm = mloc - kXWeightShift;
      alpha = ex2(m_ref - nm);
      m_ref = nm;
      ref_set = true;
    }
    // The weights go over the tile's own scores in TMEM, so only a rescale of the
    // accumulators waits for the previous tile's PV.  (A tile's scores are complete only
    // after every MMA issued before them, so tile i - 2's PV is done by now and the parity
    // wait below cannot pass on an older phase.)
    const bool resc = alpha != 1.f && l_run > 0.f;
    const bool any_resc = __any_sync(0xffffffffu, resc);
    if (i >= 1 && any_resc &&
        !__all_sync(0xffffffffu, xwait(pv_done, (uint32_t)((i - 1) & 1), a.status)))
      return false;
    tc_fence_after();
    if (any_resc) {
      const float f = resc ? alpha : 1.f;
      // the plain accumulator holds partial sums only after the first BF16 tile's PV
      // (until then its columns are the query planes)
      const uint32_t c_end = i > tl.nR ? L::C_END : L::C_OPLAIN;
#pragma unroll 1
      for (uint32_t c = L::C_OROT; c < c_end; c += 32) {
        uint32_t o[32];
        tmem_ld32_nowait(lane_base + c, o);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * f);
        tmem_st32(lane_base + c, o);
      }
      tmem_wait_st();
    }
    l_run *= alpha;
    if (m_ref == -INFINITY) m_ref = 0.f;   // no visible key yet: every weight of this tile is 0
    const float negm = -m_ref;
    // weights 2^(score - m) = ex2(raw * F - m); the row sum takes them in float32 (the split
    // terms below carry 22 or 24 bits of each)
    float lsum = 0.f;
    if (kind == kTileInt2) {
      // f16 hi / lo of the weights into this tile's score columns: column q of a plane holds
      // keys 2q, 2q + 1 (hi in columns 0..31, lo in 32..63)
      const uint32_t pcol = lane_base + L::C_S + (uint32_t)((i & 1) * kXKeys);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          const int k0 = 32 * hf + 2 * q;
          const float p0 = ex2(fmaf(sc[k0], F, negm)), p1 = ex2(fmaf(sc[k0 + 1], F, negm));
          hi[q] = half2_bits(p0, p1);
          const float2 hv = __half22float2(*reinterpret_cast<const __half2*>(&hi[q]));
          lo[q] = half2_bits(p0 - hv.x, p1 - hv.y);
          lsum += p0 + p1;
        }
        tmem_st16(pcol + (uint32_t)(16 * hf), hi);
        tmem_st16(pcol + (uint32_t)(32 + 16 * hf), lo);
      }
      tmem_wait_st();
    } else {
      // three BF16 terms of the weights (24 bits: window and chunk values are unbounded BF16):
      // hi = p with its mantissa cut to BF16, lo = the same of p - hi, lo2 = p - hi - lo, each
      // exactly a BF16 value (8 significant bits each) and hi + lo + lo2 = p exactly; a term's
      // BF16 pattern is the upper half of its float32 pattern
      const uint32_t pcol = lane_base + L::C_S + (uint32_t)((i & 1) * kXKeys);
      const uint32_t p2col = lane_base + L::C_P2 + (uint32_t)((i & 1) * (kXKeys / 2));
#pragma unroll
      for (int qt = 0; qt < 8; ++qt) {
        uint32_t hi[4], lo[4], lo2[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int k0 = 8 * qt + 2 * q;
          const float p0 = ex2(fmaf(sc[k0], F, negm)), p1 = ex2(fmaf(sc[k0 + 1], F, negm));
          const float h0 = __uint_as_float(__float_as_uint(p0) & 0xFFFF0000u);
          const float h1 = __uint_as_float(__float_as_uint(p1) & 0xFFFF0000u);
          const float r0 = p0 - h0, r1 = p1 - h1;   // exact
          const float l0 = __uint_as_float(__float_as_uint(r0) & 0xFFFF0000u);
          const float l1 = __uint_as_float(__float_as_uint(r1) & 0xFFFF0000u);
          hi[q] = prmt(__float_as_uint(h0), __float_as_uint(h1), 0x7632u);
          lo[q] = prmt(__float_as_uint(l0), __float_as_uint(l1), 0x7632u);
          lo2[q] = prmt(__float_as_uint(r0 - l0), __float_as_uint(r1 - l1), 0x7632u);
          lsum += p0 + p1;
        }
        tmem_st4(pcol + (uint32_t)(4 * qt), hi);
        tmem_st4(pcol + (uint32_t)(32 + 4 * qt), lo);
        tmem_st4(p2col + (uint32_t)(4 * qt), lo2);
      }
      tmem_wait_st();
    }
    l_run += lsum;
    return true;
  };

  int raw_issued = 0;     // copying warp: INT2 tiles [0, raw_issued) requested
  int raw_done = 0;       // its lane 0: INT2 tiles [0, raw_done) arrived (waited on)
  // ---------------- preamble: zero the output accumulators, query planes, first pages
  if (warp < 4) {
    uint32_t z[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) z[k] = 0u;
#pragma unroll 1
    for (uint32_t c = L::C_OROT; c < L::C_OPLAIN; c += 32) tmem_st32(lane_base + c, z);
    if (tl.nR > 0) write_q_rot();
    write_q_plain();
    tmem_wait_st();
  } else if (warp == 4 && !use_prep) {
    // the pages of the first NRAW - 1 tiles (the loop requests tile j + NRAW - 1 at tile j)
#pragma unroll 1
    for (int t = 0; t < L::NRAW - 1 && t < tl.nR; ++t) {
      int pg[kMaxBlk];
      tile_pages(t, pg);
      if (lane == 0) issue_raw(t, pg);
    }
    raw_issued = min(L::NRAW - 1, tl.nR);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // ---------------- pipeline: the roles meet only at mbarriers.  The MMA thread issues the
  // scores of tile j as soon as tile j is unpacked (the softmax may still be on tile j - 1)
  // and the PV of tile j - 1 when its weights are in place.
  bool aborted = false;
  if (warp < 4) {
    for (int i = 0; i < n_tiles; ++i) {
      const bool ok = __all_sync(0xffffffffu, *abort_flag == 0) && softmax_tile(i);
      if (!ok) {
        *abort_flag = 1;
        aborted = true;
        break;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[i & 1]);
    }
  } else if (warp < 8) {
    int copies_issued = 0;   // unpacked form, warp 4 lane 0: tiles [0, copies_issued) requested
    int copies_done = 0;     // tiles [0, copies_done) known to have landed (their stage was freed since)
    for (int j = 0; j < n_tiles; ++j) {
      // stage j % NST was last read by tile j - NST's MMAs
      const bool ok = j < L::NST || xwait(&kv_empty[j % L::NST], (uint32_t)(((j / L::NST) - 1) & 1), a.status);
      // one named barrier per tile: every thread is done with tile j - 1 (so its raw buffer
      // may take tile j + NRAW - 1), and all agree on whether to stop
      if (unpack_bar_any(!ok || *abort_flag != 0)) {
        *abort_flag = 1;
        aborted = true;
        break;
      }
      if (j >= L::NST) copies_done = j - L::NST + 1;
      if (use_prep) {
        // the tile's image: one bulk copy into its stage by warp 4 lane 0, whose arrival
        // carries the bytes; warps 5-7 arrive at once
        if (lane == 0) {
          uint64_t* bar = &kv_full[j % L::NST];
          if (warp == 4) {
            const int pj = j < tl.nR ? j : (j < tl.nR + tl.nW ? a.prep_tiles + (j - tl.nR)
                                                              : a.prep_tiles + a.prep_wt + (j - tl.nR - tl.nW));
            mbar_arrive_expect_tx(bar, (uint32_t)L::STAGE);
            bulk_g2s(smem + L::ST0 + (j % L::NST) * L::STAGE,
                     a.prep + (((size_t)b * g.Hkv + kvh) * (a.prep_tiles + a.prep_wt + a.prep_ct) + pj) * L::STAGE,
                     (uint32_t)L::STAGE, bar);
            copies_issued = j + 1;
          } else {
            mbar_arrive(bar);
          }
        }
        continue;
      }
      if (warp == 4 && !use_prep && j + L::NRAW - 1 < tl.nR) {
        int pg[kMaxBlk];
        tile_pages(j + L::NRAW - 1, pg);
        if (lane == 0) issue_raw(j + L::NRAW - 1, pg);
        raw_issued = j + L::NRAW;
      }
      // a late page flags the CTA to stop at the next barrier (every thread still reaches it)
      if (unpack(j)) {
        if (j < tl.nR) raw_done = j + 1;
      } else {
        *abort_flag = 1;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&kv_full[j % L::NST]);
    }
    // no bulk copy may still be writing this CTA's shared memory when it exits (bounded waits;
    // a stage copy not yet known to have landed is the last on its stage, so its phase parity
    // is unambiguous)
    if (u == 0) {
      for (int t = raw_done; t < raw_issued; ++t)
        (void)mbar_wait_bounded(&raw_full[t % L::NRAW], (uint32_t)((t / L::NRAW) & 1), nullptr);
      for (int t = copies_done; t < copies_issued; ++t)
        (void)mbar_wait_bounded(&kv_full[t % L::NST], (uint32_t)((t / L::NST) & 1), nullptr);
    }
  } else if (warp == 8 && lane == 0) {
    // MMA issue: the scores of tile qk (its stage unpacked; its S buffer, which holds tile
    // qk - 2's weights, free once that tile's PV is issued: the MMAs run in issue order) and
    // the PV of tile pv (its weights in place), whichever is ready first
    int qk = 0, pv = 0;
    int last_commit = -1;   // 0: s_full of tile qk - 1, 1: pv_done of tile pv - 1
    // the timer is read only while no MMA can be issued (a read on every issue cost 1.4 %)
    uint64_t t_idle = 0;   // start of the current stretch without progress (0: none)
    while (pv < n_tiles) {
      bool progressed = false;
      if (qk < n_tiles && pv >= qk - 1 &&
          mbar_try_wait(&kv_full[qk % L::NST], (uint32_t)((qk / L::NST) & 1))) {
        tc_fence_after();
        issue_qk(qk);
        tc_commit(&s_full[qk & 1]);
        last_commit = 0;
        ++qk;
        progressed = true;
      }
      if (pv < qk && mbar_try_wait(&p_full[pv & 1], (uint32_t)((pv >> 1) & 1))) {
        tc_fence_after();
        issue_pv(pv);
        tc_commit(pv_done);
        if (pv + L::NST < n_tiles) tc_commit(&kv_empty[pv % L::NST]);
        last_commit = 1;
        ++pv;
        progressed = true;
      }
      if (progressed) {
        t_idle = 0;
        continue;
      }
      __nanosleep(32);
      const uint64_t now = globaltimer_ns();
      if (t_idle == 0) t_idle = now;
      if (*abort_flag || now - t_idle > kWaitLimitNs) {
        if (!*abort_flag) flag_error(a.status, kDevTimeout);
        *abort_flag = 1;
        aborted = true;
        break;
      }
    }
    if (aborted) {
      // drain: the last commit covers every MMA issued before it
      if (last_commit == 1) (void)xwait(pv_done, (uint32_t)((pv - 1) & 1), nullptr);
      else if (last_commit == 0) (void)xwait(&s_full[(qk - 1) & 1], (uint32_t)(((qk - 1) >> 1) & 1), nullptr);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (*abort_flag) {
    if (warp == 8) tmem_dealloc(tmem, L::TMEM_COLS);
    return;
  }
  (void)aborted;

  // ---------------- epilogue: out = O_plain / l + (y / l) R_V^T.  y / l goes to TMEM as f16 hi and
  // lo planes over the dead score columns (the A operand), R_V's planes arrive by one bulk copy
  // (the B operand), and three MMAs per K step (hi hi, hi lo, lo hi) leave y R_V^T / l in the
  // rotated accumulator's columns.  A CTA without INT2 tiles has a zero rotated accumulator and
  // skips all of it.
  bool ok = true;
  if (warp < 8) {
    ok = __all_sync(0xffffffffu, xwait(pv_done, (uint32_t)((n_tiles - 1) & 1), a.status));
    tc_fence_after();
  }
  float* linv = reinterpret_cast<float*>(smem + L::LINV);
  const int half = (tid >> 7) & 1;
  constexpr int NJ = D / 2;
  const int j0 = half * NJ;
  if (warp < 4) linv[r] = l_run > 0.f ? 1.f / l_run : 0.f;
  // every MMA has completed (or the CTA stores nothing): the shared memory below is free
  const bool rotated = __syncthreads_and(ok) && tl.nR > 0;
  if (rotated && tid == 0) {
    mbar_arrive_expect_tx(epi_copy, (uint32_t)L::RP_BYTES);
    bulk_g2s(smem + L::RP, a.ws + a.rvp_off + (g.rph ? (size_t)kvh * L::RP_BYTES : 0), (uint32_t)L::RP_BYTES,
             epi_copy);
  }
  if (rotated && warp < 8) {
    const float li = linv[r];
    uint32_t oz[32];
    tmem_ld32_nowait(lane_base + L::C_OZ, oz);
    tmem_wait_ld();
#pragma unroll
    for (int cb = 0; cb < NJ / 32; ++cb) {
      uint32_t o[32];
      tmem_ld32_nowait(lane_base + L::C_OROT + (uint32_t)(j0 + 32 * cb), o);
      tmem_wait_ld();
      const int gidx = (j0 >> 5) + cb;   // this block's group
      float zsel = 0.f;
#pragma unroll
      for (int gg = 0; gg < G; ++gg)
        zsel = gg == gidx ? __uint_as_float(oz[gg]) + __uint_as_float(oz[G + gg]) : zsel;
      const float zv = zsel * pow2f(-a.k_exp_V);
      uint32_t hi[16], lo[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        const int ch = j0 + 32 * cb + 2 * q;
        const float y0 = fmaf(__uint_as_float(o[2 * q]), pow2f(10 - slot_pos((ch % 64) / 8) - a.k_exp_V), zv) * li;
        const float y1 =
            fmaf(__uint_as_float(o[2 * q + 1]), pow2f(10 - slot_pos(((ch + 1) % 64) / 8) - a.k_exp_V), zv) * li;
        hi[q] = half2_bits(y0, y1);
        const float2 hf = __half22float2(*reinterpret_cast<const __half2*>(&hi[q]));
        lo[q] = half2_bits(y0 - hf.x, y1 - hf.y);
      }
      tmem_st16(lane_base + L::C_S + (uint32_t)(j0 / 2 + 16 * cb), hi);
      tmem_st16(lane_base + L::C_S + (uint32_t)(D / 2 + j0 / 2 + 16 * cb), lo);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (rotated && warp == 8 && lane == 0) {
    const bool okc = mbar_wait_bounded(epi_copy, 0, a.status);
    tc_fence_after();
    if (okc) {
      const uint64_t dRP = smem_desc_sw128(smem_u32(smem) + L::RP);
      const uint32_t idesc = idesc_f16_f32(kXRows, D);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t bk = (uint32_t)((kk >> 2) * D * 128 + (kk & 3) * 32);
        const uint32_t a_hi = tmem + L::C_S + (uint32_t)(8 * kk), a_lo = a_hi + (uint32_t)(D / 2);
        tc_mma_ts(tmem + L::C_OROT, a_hi, dadd(dRP, bk), idesc, kk ? 1u : 0u);
        tc_mma_ts(tmem + L::C_OROT, a_hi, dadd(dRP, (uint32_t)(D * D * 2) + bk), idesc, 1u);
        tc_mma_ts(tmem + L::C_OROT, a_lo, dadd(dRP, bk), idesc, 1u);
      }
    } else {
      (void)mbar_wait_bounded(epi_copy, 0, nullptr);   // the copy lands before the CTA exits
    }
    tc_commit(epi_mma);
  }
  if (warp < 8) {
    bool okm = ok;
    if (rotated) {
      okm = __all_sync(0xffffffffu, xwait(epi_mma, 0, a.status));
      tc_fence_after();
    }
    const float li = linv[r];
    float acc[NJ];
#pragma unroll
    for (int cb = 0; cb < NJ / 32; ++cb) {
      uint32_t o[32], y[32];
      tmem_ld32_nowait(lane_base + L::C_OPLAIN + (uint32_t)(j0 + 32 * cb), o);
      if (rotated) tmem_ld32_nowait(lane_base + L::C_OROT + (uint32_t)(j0 + 32 * cb), y);
      tmem_wait_ld();
#pragma unroll
      for (int k = 0; k < 32; ++k)
        acc[32 * cb + k] = rotated ? fmaf(__uint_as_float(o[k]), li, __uint_as_float(y[k])) : __uint_as_float(o[k]) * li;
    }
    if (!okm || !row_ok) {
      // nothing to store
    } else if (a.out_dtype == kDtypeF32) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + qrow * D + j0);
#pragma unroll
      for (int j4 = 0; j4 < NJ / 4; ++j4)
        dst[j4] = make_float4(acc[4 * j4], acc[4 * j4 + 1], acc[4 * j4 + 2], acc[4 * j4 + 3]);
    } else {
      uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + qrow * D + j0);
#pragma unroll
      for (int j8 = 0; j8 < NJ / 8; ++j8)
        dst[j8] = make_uint4(pack_bf162(acc[8 * j8], acc[8 * j8 + 1]), pack_bf162(acc[8 * j8 + 2], acc[8 * j8 + 3]),
                             pack_bf162(acc[8 * j8 + 4], acc[8 * j8 + 5]), pack_bf162(acc[8 * j8 + 6], acc[8 * j8 + 7]));
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 8) tmem_dealloc(tmem, L::TMEM_COLS);
}

template <int D>
int launch_extend_d(const ExtendArgs& a, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long rows = (long long)a.total_tokens * a.g.Hq;
  const size_t qsm = QrPlan<D>::SMEM;
  cudaError_t e = ensure_smem_limit(extend_qrot_kernel<D>, qsm);
  if (e != cudaSuccess) return (int)e;
  // one rotation per kv head: grid.y = kv heads, each CTA 128 / gq tokens of its head's query rows
  const int heads = a.g.rph ? a.g.Hkv : 1;
  const long long per = a.g.rph ? 128 / a.g.gq() : 128;
  const long long units = a.g.rph ? (long long)a.total_tokens : rows;
  const unsigned qgrid = (unsigned)((units + per - 1) / per) + 1;
  if (a.prep) {
    const size_t usm = XLayout<D>::STAGE + XLayout<D>::RAW_BYTES + 1024;
    if ((e = ensure_smem_limit(extend_unpack_kernel<D>, usm)) != cudaSuccess) return (int)e;
    const unsigned tiles = (unsigned)(a.prep_tiles + a.prep_wt + a.prep_ct);
    extend_unpack_kernel<D><<<dim3(tiles, (unsigned)a.g.Hkv, (unsigned)a.batch), 128, usm, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return (int)e;
  }
  extend_qrot_kernel<D><<<dim3(qgrid, heads), 128, qsm, s>>>(a);
  if ((e = cudaGetLastError()) != cudaSuccess) return (int)e;
  auto kern = a.prep ? extend_attn_kernel<D, true> : extend_attn_kernel<D, false>;
  e = ensure_smem_limit(kern, XLayout<D>::SMEM);
  if (e != cudaSuccess) return (int)e;
  const int tq = kXRows / a.g.gq();
  dim3 grid((unsigned)((a.max_chunk + tq - 1) / tq), (unsigned)a.g.Hkv, (unsigned)a.batch);
  kern<<<grid, kXThreads, XLayout<D>::SMEM, s>>>(a);
  return (int)cudaGetLastError();
}

}  // namespace

// workspace: R_V's f16 hi and lo planes ([Hkv][2][D][D] with a rotation per kv head, else
// [2][D][D]; the size of a float32 D x D per rotation), then q R_K per row
size_t extend_workspace_bytes(const Geom& g, long long total_tokens) {
  const size_t rvp = ((size_t)(g.rph ? g.Hkv : 1) * g.D * g.D * 4 + 255) & ~size_t(255);
  return rvp + (size_t)total_tokens * g.Hq * g.D * 4;
}

void extend_ws_offsets(const Geom& g, size_t* rvp_off, size_t* qrot_off) {
  *rvp_off = 0;
  *qrot_off = ((size_t)(g.rph ? g.Hkv : 1) * g.D * g.D * 4 + 255) & ~size_t(255);
}

size_t extend_prep_tile_bytes(int D) { return D == 128 ? XLayout<128>::STAGE : XLayout<64>::STAGE; }

long long extend_prep_tiles(const Geom& g, long long max_prefix) {
  const long long hist_end = max_prefix - g.W > g.S ? max_prefix - g.W : g.S;
  return hist_end > g.S ? (hist_end - 1) / 64 - g.S / 64 + 1 : 0;
}

int extend_prep_window_tiles(const Geom& g) { return (g.S + g.W + 63) / 64; }

long long extend_prep_chunk_tiles(const Geom& g, long long max_chunk) {
  // the attention grid covers ceil(max_chunk / tq) query tiles of tq tokens, so a chunk may hold
  // up to that many tokens (more is flagged)
  const long long tq = kXRows / g.gq();
  return ((max_chunk + tq - 1) / tq * tq + 63) / 64;
}

int launch_extend(const ExtendArgs& a, void* stream) {
  if (a.total_tokens == 0 || a.batch == 0 || a.max_chunk == 0) return 0;
  if (a.g.D == 128) return launch_extend_d<128>(a, stream);
  return launch_extend_d<64>(a, stream);
}

}  // namespace oscar
