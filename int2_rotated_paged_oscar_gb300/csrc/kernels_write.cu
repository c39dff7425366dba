// Write path of the OSCAR INT2 paged cache: prefill/extend, eviction of ring
// tokens, and the single-token decode append.
//
// Source: OSCAR technical summary (gist.science), section 2.2 B -- history is
// stored in INT2 after the fixed rotation and clipping, sink and recent tokens
// stay BF16; arXiv abstract -- fused write kernel, fixed per-layer rotations.
// The quantiser (per token/head/group of 32 channels, asymmetric min/max, BF16
// scale and zero, round-to-nearest-even codes clamped to [0, 3]) and the code
// layouts are the ones documented in include/oscar.h.
//
// Lane l of a warp owns output channels [l*D/32, (l+1)*D/32) of a row.  The
// rotation y_j = sum_i x_i R[i][j] runs in float32 in one canonical order used
// by every kernel of this file: four partial sums over the input quarters
// i in [kD/4, (k+1)D/4), each one FMA per term in increasing i starting from
// zero, added as ((c0 + c1) + c2) + c3.  The prefill, eviction and append paths
// therefore produce identical codes for the same BF16 input, whichever way
// they spread the four chains over warps.  The Hadamard-only variant replaces
// the dense product by a fast Walsh-Hadamard transform followed by the
// bit-reversal gather.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "oscar_internal.h"

namespace oscar {
namespace {

#include "q_rotate.cuh"

constexpr int kWarpsPerCta = 8;

// ------------------------------------------------------------------ row helpers
template <int D>
struct RowPtrs {
  uint8_t* codes;   // start of the code row
  uint32_t* sz;     // start of the (scale, zero) row: D/32 uint32
};

__device__ __forceinline__ float load_in(const void* base, int dtype, size_t idx) {
  if (dtype == kDtypeBF16) {
    const uint16_t v = static_cast<const uint16_t*>(base)[idx];
    return __uint_as_float(static_cast<uint32_t>(v) << 16);
  }
  return static_cast<const float*>(base)[idx];
}

__device__ __forceinline__ uint16_t to_bf16_bits(float x) {
  __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t*>(&h);
}

// Rotate x (D floats in shared memory, one warp's buffer) by R (global or
// shared, row-major), or by H_Had . P_br when hadamard != 0.  Returns this
// lane's D/32 outputs.
template <int D>
__device__ __forceinline__ void rotate_row(const float* xs, const float* R, int hadamard, float (&y)[D / 32],
                                           float* scratch) {
  constexpr int C = D / 32;
  const int lane = threadIdx.x & 31;
  if (!hadamard) {
    float ch[4][C];
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int c = 0; c < C; ++c) ch[k][c] = 0.f;
#pragma unroll 8
    for (int i = 0; i < D / 4; ++i) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int ii = k * (D / 4) + i;
        const float xi = xs[ii];
        const float* r = R + (size_t)ii * D + lane * C;
#pragma unroll
        for (int c = 0; c < C; ++c) ch[k][c] = fmaf(xi, r[c], ch[k][c]);
      }
    }
#pragma unroll
    for (int c = 0; c < C; ++c) y[c] = ((ch[0][c] + ch[1][c]) + ch[2][c]) + ch[3][c];
    return;
  }
  // Fast Walsh-Hadamard transform in natural (Sylvester) order: lane holds
  // elements lane*C + c; butterflies with partner distance < C stay in
  // registers, larger ones use shuffles.
  float v[C];
#pragma unroll
  for (int c = 0; c < C; ++c) v[c] = xs[lane * C + c];
#pragma unroll
  for (int hlen = 1; hlen < C; hlen <<= 1) {
#pragma unroll
    for (int c = 0; c < C; ++c) {
      if ((c & hlen) == 0) {
        const float a = v[c], b = v[c + hlen];
        v[c] = a + b;
        v[c + hlen] = a - b;
      }
    }
  }
#pragma unroll
  for (int lm = 1; lm < 32; lm <<= 1) {
    const bool upper = (lane & lm) != 0;
#pragma unroll
    for (int c = 0; c < C; ++c) {
      const float o = __shfl_xor_sync(0xffffffffu, v[c], lm);
      v[c] = upper ? (o - v[c]) : (v[c] + o);
    }
  }
  const float inv = D == 64 ? 0.125f : 0.08838834764831845f;  // 1/sqrt(D) rounded to float32
#pragma unroll
  for (int c = 0; c < C; ++c) scratch[lane * C + c] = v[c] * inv;
  __syncwarp();
  // (x H P_br)_j = (x H)_{br(j)}
  constexpr int nbits = D == 64 ? 6 : 7;
#pragma unroll
  for (int c = 0; c < C; ++c) {
    const int j = lane * C + c;
    const int br = __brev(j) >> (32 - nbits);
    y[c] = scratch[br];
  }
  __syncwarp();
}

// Clip, quantise and pack one rotated row into its page slot.
template <int D>
__device__ __forceinline__ void quant_pack_store(const float (&y_in)[D / 32], float clip, bool is_v,
                                                 uint8_t* row_codes, uint32_t* row_sz, uint8_t* code_scratch) {
  constexpr int C = D / 32;
  constexpr int LPG = 32 / C;  // lanes per group of 32 channels
  const int lane = threadIdx.x & 31;
  float y[C];
  float mn = INFINITY, mx = -INFINITY;
#pragma unroll
  for (int c = 0; c < C; ++c) {
    y[c] = fminf(fmaxf(y_in[c], -clip), clip);
    mn = fminf(mn, y[c]);
    mx = fmaxf(mx, y[c]);
  }
#pragma unroll
  for (int m = 1; m < LPG; m <<= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, m));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
  }
  const uint16_t zb = to_bf16_bits(mn);
  const uint16_t sb = to_bf16_bits((mx - mn) / 3.0f);
  const float z = __uint_as_float(static_cast<uint32_t>(zb) << 16);
  const float s = __uint_as_float(static_cast<uint32_t>(sb) << 16);
#pragma unroll
  for (int c = 0; c < C; ++c) {
    int code = 0;
    if (s > 0.f) {
      const float t = (y[c] - z) / s;
      code = min(3, max(0, __float2int_rn(t)));
    }
    code_scratch[lane * C + c] = static_cast<uint8_t>(code);
  }
  __syncwarp();
  constexpr int WORDS = D / 16;
  if (lane < WORDS) {
    uint32_t word = 0;
    if (!is_v) {
      constexpr int WPL = D / 64;  // words per lane-group tig
      const int tig = lane / WPL, w = lane % WPL;
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const int p8 = 8 * w + x;
        const int ch = 32 * (p8 >> 2) + 16 * ((p8 >> 1) & 1) + 8 * (p8 & 1) + 2 * tig;
        word |= static_cast<uint32_t>(code_scratch[ch]) << (2 * x);
        word |= static_cast<uint32_t>(code_scratch[ch + 1]) << (16 + 2 * x);
      }
    } else {
      constexpr int PER = D / 64;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int hw = 2 * lane + half;
#pragma unroll
        for (int sl = 0; sl < 8; ++sl) {
          const int ch = 64 * (hw % PER) + 8 * sl + hw / PER;
          word |= static_cast<uint32_t>(code_scratch[ch]) << (16 * half + 2 * sl);
        }
      }
    }
    reinterpret_cast<uint32_t*>(row_codes)[lane] = word;
  }
  if (lane % LPG == 0) {
    row_sz[lane / LPG] = static_cast<uint32_t>(sb) | (static_cast<uint32_t>(zb) << 16);
  }
  __syncwarp();
}

template <int D>
__device__ __forceinline__ void history_row_ptrs(const WriteArgs& a, int page, int slot, int h, bool is_v,
                                                 uint8_t** codes, uint32_t** sz) {
  const Geom& g = a.g;
  uint8_t* blk = a.pool + (((size_t)a.layer * g.num_pages + page) * g.Hkv + h) * g.block_bytes();
  const size_t c_off = is_v ? g.v_codes_off() : 0;
  const size_t s_off = is_v ? g.v_sz_off() : g.k_sz_off();
  *codes = blk + c_off + (size_t)slot * (D / 4);
  *sz = reinterpret_cast<uint32_t*>(blk + s_off + (size_t)slot * (D / 8));
}

__device__ __forceinline__ uint16_t* window_row(const WriteArgs& a, int req, int h, bool is_v, int wslot) {
  const Geom& g = a.g;
  const size_t base = ((size_t)a.layer * g.max_req + req) * g.slab_req_elems();
  return a.slab + base + (((size_t)h * 2 + (is_v ? 1 : 0)) * g.window() + wslot) * g.D;
}

__device__ __forceinline__ int window_slot(int t, int S, int W) { return t < S ? t : S + (t - S) % W; }

// Page holding history token t of request b, or -1 (flagged) if unmapped.
__device__ __forceinline__ int history_page(const WriteArgs& a, int b, int t) {
  const Geom& g = a.g;
  const int lp = t / g.P;
  int page = -1;
  if (lp < a.bt_stride && lp < g.max_pages_per_req) page = a.block_table[(size_t)b * a.bt_stride + lp];
  if (page < 0 || page >= g.num_pages) {
    if ((threadIdx.x & 31) == 0) flag_error(a.status, kDevBadPage);
    return -1;
  }
  return page;
}

// Quantise the row held in xs (float32, D values) into history slot t of request b.
template <int D>
__device__ void store_history(const WriteArgs& a, int b, int t, int h, bool is_v, const float* xs, const float* R,
                              uint8_t* code_scratch, float* fscratch) {
  const Geom& g = a.g;
  const int lp = t / g.P;
  int page = -1;
  if (lp < a.bt_stride && lp < g.max_pages_per_req) page = a.block_table[(size_t)b * a.bt_stride + lp];
  if (page < 0 || page >= g.num_pages) {
    if ((threadIdx.x & 31) == 0) flag_error(a.status, kDevBadPage);
    return;
  }
  float y[D / 32];
  rotate_row<D>(xs, R, a.hadamard, y, fscratch);
  uint8_t* codes;
  uint32_t* sz;
  history_row_ptrs<D>(a, page, t % g.P, h, is_v, &codes, &sz);
  quant_pack_store<D>(y, is_v ? a.clip_V : a.clip_K, is_v, codes, sz, code_scratch);
}

struct WarpSmem {
  float x[128];
  float f[128];
  uint8_t codes[128];
};

// ------------------------------------------------------------------ prefill / extend
// grid (ctas, 2): blockIdx.y selects K (0) or V (1).  The CTA keeps R in shared
// memory; each warp takes kRowsPerPass (token, kv head) rows at a time and
// rotates them together so every R element read from shared memory feeds
// kRowsPerPass FMAs.
constexpr int kRowsPerPass = 4;

template <int D>
struct WriteSmem {
  float x[kWarpsPerCta][kRowsPerPass][D];
  float scratch[kWarpsPerCta][D];  // FWHT gather buffer
  int meta[kWarpsPerCta][kRowsPerPass][3];  // (request, token, kv head) of history rows
  uint8_t codes[kWarpsPerCta][D];
};

template <int D>
__global__ void __launch_bounds__(kWarpsPerCta * 32, 2) write_kernel(WriteArgs a) {
  constexpr int C = D / 32;
  extern __shared__ __align__(16) float wsm[];
  pdl_wait();  // the eviction before it reads ring rows this kernel overwrites
  float* Rs = wsm;                                                  // [D][D]
  WriteSmem<D>& sm = *reinterpret_cast<WriteSmem<D>*>(wsm + D * D);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool is_v = blockIdx.y == 1;
  const Geom& g = a.g;
  const void* src = is_v ? a.V : a.K;
  // one rotation per layer: rows (token, kv head) of every head; one per kv head: this CTA
  // takes the rows of kv head blockIdx.z with that head's rotation
  const int hz = g.rph ? (int)blockIdx.z : 0;
  if (!a.hadamard) {  // the Hadamard-only rotation has no matrix (R_K, R_V are null)
    const float4* Rg = reinterpret_cast<const float4*>((is_v ? a.R_V : a.R_K) + (size_t)hz * g.rot_stride());
    float4* R4 = reinterpret_cast<float4*>(Rs);
    for (int i = threadIdx.x; i < D * D / 4; i += blockDim.x) R4[i] = Rg[i];
  }
  __syncthreads();
  const long long rows = g.rph ? (long long)a.total_tokens : (long long)a.total_tokens * g.Hkv;
  const long long stride = (long long)gridDim.x * kWarpsPerCta * kRowsPerPass;
  for (long long base = ((long long)blockIdx.x * kWarpsPerCta + warp) * kRowsPerPass; base < rows; base += stride) {
    unsigned hist = 0;  // bit r: row r goes to an INT2 page
#pragma unroll 1
    for (int r = 0; r < kRowsPerPass; ++r) {
      const long long item = base + r;
      if (item >= rows) continue;
      const int row = g.rph ? static_cast<int>(item) : static_cast<int>(item / g.Hkv);
      const int h = g.rph ? hz : static_cast<int>(item % g.Hkv);
      int lo = 0, hi = a.batch - 1;  // request of this row: largest b with cu_seqlens[b] <= row
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.cu_seqlens[mid] <= row) lo = mid; else hi = mid - 1;
      }
      const int b = lo;
      const int t0 = a.start_pos[b];
      const int len = a.cu_seqlens[b + 1] - a.cu_seqlens[b];
      const int t = t0 + (row - a.cu_seqlens[b]);
      const int n1 = t0 + len;
      if (t0 < 0 || n1 > g.max_pages_per_req * g.P) {
        if (lane == 0) flag_error(a.status, kDevBadLen);
        continue;
      }
      const size_t in_base = ((size_t)row * g.Hkv + h) * D;
      if (t >= g.S && t < n1 - g.W) {
        hist |= 1u << r;
        if (lane == 0) {
          sm.meta[warp][r][0] = b;
          sm.meta[warp][r][1] = t;
          sm.meta[warp][r][2] = h;
        }
        for (int i = lane; i < D; i += 32) sm.x[warp][r][i] = load_in(src, a.dtype, in_base + i);
      } else {
        const int req = a.req_slot[b];
        if (req < 0 || req >= g.max_req) {
          if (lane == 0) flag_error(a.status, kDevBadSlot);
          continue;
        }
        uint16_t* dst = window_row(a, req, h, is_v, window_slot(t, g.S, g.W));
        for (int i = lane; i < D; i += 32) dst[i] = to_bf16_bits(load_in(src, a.dtype, in_base + i));
      }
    }
    __syncwarp();
    if (!hist) continue;
    float y[kRowsPerPass][C];
    if (a.hadamard) {
#pragma unroll
      for (int r = 0; r < kRowsPerPass; ++r)
        if (hist >> r & 1) rotate_row<D>(sm.x[warp][r], nullptr, 1, y[r], sm.scratch[warp]);
    } else {
      float ch[kRowsPerPass][4][C];
#pragma unroll
      for (int r = 0; r < kRowsPerPass; ++r)
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int c = 0; c < C; ++c) ch[r][k][c] = 0.f;
#pragma unroll 2
      for (int i = 0; i < D / 4; ++i) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int ii = k * (D / 4) + i;
          float rv[C];
          if constexpr (C == 4) {
            const float4 q4 = *reinterpret_cast<const float4*>(Rs + ii * D + lane * 4);
            rv[0] = q4.x; rv[1] = q4.y; rv[2] = q4.z; rv[3] = q4.w;
          } else {
            const float2 q2 = *reinterpret_cast<const float2*>(Rs + ii * D + lane * 2);
            rv[0] = q2.x; rv[1] = q2.y;
          }
#pragma unroll
          for (int r = 0; r < kRowsPerPass; ++r) {
            const float xi = sm.x[warp][r][ii];
#pragma unroll
            for (int c = 0; c < C; ++c) ch[r][k][c] = fmaf(xi, rv[c], ch[r][k][c]);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < kRowsPerPass; ++r)
#pragma unroll
        for (int c = 0; c < C; ++c) y[r][c] = ((ch[r][0][c] + ch[r][1][c]) + ch[r][2][c]) + ch[r][3][c];
    }
#pragma unroll
    for (int r = 0; r < kRowsPerPass; ++r) {
      if (!(hist >> r & 1)) continue;
      const int rb = sm.meta[warp][r][0], rt = sm.meta[warp][r][1], rh = sm.meta[warp][r][2];
      const int page = history_page(a, rb, rt);
      if (page < 0) continue;
      uint8_t* codes;
      uint32_t* sz;
      history_row_ptrs<D>(a, page, rt % g.P, rh, is_v, &codes, &sz);
      quant_pack_store<D>(y[r], is_v ? a.clip_V : a.clip_K, is_v, codes, sz, sm.codes[warp]);
    }
    __syncwarp();
  }
}

// ------------------------------------------------------------------ prefill / extend, rotation H_Had . P_br
// The Hadamard-only write (no matrix).  The row x of a (token, kv head) is held by a
// quad of lanes: quad lane q (0..3) holds elements [q E, q E + E), E = D/4.  The fast
// Walsh-Hadamard transform (Sylvester order) runs its log2(E) low stages in registers
// and its two top stages across the quad (xor shuffles); y = x H / sqrt(D).  The
// bit-reversal gather P_br moves no data: element i = q E + c is output channel
// j = br(i) = 4 br(c) + br2(q), so quantisation group gi is the register set
// { c : c mod G = br(gi) } (eight registers per quad lane) and its channel
// u = 4 br3(c / G) + br2(q).  Group min/max: eight registers, then two quad
// shuffles.  Four codes fill one byte of a page code word; the bytes meet in a
// per-warp row buffer, from which each quad lane stores a quarter of the row.
// A warp takes 8 rows per pass; the request lookup is cached per lane.
constexpr int kFwhtWarps = 8;

__device__ __forceinline__ int brev_bits(int x, int nbits) { return nbits ? (int)(__brev((unsigned)x) >> (32 - nbits)) : 0; }

template <int D>
__global__ void __launch_bounds__(kFwhtWarps * 32) write_fwht_kernel(WriteArgs a) {
  pdl_wait();  // the eviction before it reads ring rows this kernel overwrites
  constexpr int E = D / 4, G = D / 32, NG = D == 128 ? 2 : 1;  // NG = log2(G)
  constexpr int WPQ = D / 64;                                    // code words per quad lane
  __shared__ __align__(16) uint8_t cbuf[kFwhtWarps][8][D / 4];  // [warp][row of the pass]: the row's code words
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = lane & 3, rl = lane >> 2;
  const bool is_v = blockIdx.y == 1;
  const Geom& g = a.g;
  const float clip = is_v ? a.clip_V : a.clip_K;
  // the page size is a power of two (checked by the host); n_kv_heads usually is
  const bool hkv_pow2 = (g.Hkv & (g.Hkv - 1)) == 0;
  const int hkv_sh = __ffs(g.Hkv) - 1, p_sh = __ffs(g.P) - 1;
  const long long rows = (long long)a.total_tokens * g.Hkv;
  const long long step = (long long)gridDim.x * kFwhtWarps * 8;
  int cb = 0, cb0 = 0, cb1 = -1, ct0 = 0;  // cached request: tokens [cb0, cb1) of request cb, start_pos ct0
  for (long long base = ((long long)blockIdx.x * kFwhtWarps + warp) * 8; base < rows; base += step) {
    const long long r = base + rl;
    const bool live = r < rows;
    const int token = live ? static_cast<int>(hkv_pow2 ? r >> hkv_sh : r / g.Hkv) : 0;
    const int h = live ? static_cast<int>(hkv_pow2 ? r & (g.Hkv - 1) : r % g.Hkv) : 0;
    float v[E];
    const size_t in_base = ((size_t)token * g.Hkv + h) * D + (size_t)q * E;
    if (!live) {
#pragma unroll
      for (int c = 0; c < E; ++c) v[c] = 0.f;
    } else if (a.dtype == kDtypeBF16) {
      const uint4* p = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(is_v ? a.V : a.K) + in_base);
#pragma unroll
      for (int k = 0; k < E / 8; ++k) {
        const uint4 w = p[k];
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[8 * k + 2 * e] = __uint_as_float(ww[e] << 16);
          v[8 * k + 2 * e + 1] = __uint_as_float(ww[e] & 0xFFFF0000u);
        }
      }
    } else {
      const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(is_v ? a.V : a.K) + in_base);
#pragma unroll
      for (int k = 0; k < E / 4; ++k) {
        const float4 w = p[k];
        v[4 * k] = w.x; v[4 * k + 1] = w.y; v[4 * k + 2] = w.z; v[4 * k + 3] = w.w;
      }
    }
    int kind = 0, t = 0;  // kind 1: INT2 history row, 2: BF16 window row
    if (live) {
      if (token < cb0 || token >= cb1) {
        int lo = 0, hi = a.batch - 1;  // largest b with cu_seqlens[b] <= token
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (a.cu_seqlens[mid] <= token) lo = mid; else hi = mid - 1;
        }
        cb = lo;
        cb0 = a.cu_seqlens[cb];
        cb1 = a.cu_seqlens[cb + 1];
        ct0 = a.start_pos[cb];
      }
      t = ct0 + (token - cb0);
      const int n1 = ct0 + (cb1 - cb0);
      if (ct0 < 0 || n1 > g.max_pages_per_req * g.P) {
        if (q == 0) flag_error(a.status, kDevBadLen);
      } else {
        kind = (t >= g.S && t < n1 - g.W) ? 1 : 2;
      }
    }
    int page = -1;  // read now, used after the transform
    if (kind == 1) {
      const int lp = t >> p_sh;
      if (lp < a.bt_stride && lp < g.max_pages_per_req) page = a.block_table[(size_t)cb * a.bt_stride + lp];
    }
    if (kind == 2) {
      const int req = a.req_slot[cb];
      if (req < 0 || req >= g.max_req) {
        if (q == 0) flag_error(a.status, kDevBadSlot);
      } else {
        uint4* dst = reinterpret_cast<uint4*>(window_row(a, req, h, is_v, window_slot(t, g.S, g.W)) + q * E);
#pragma unroll
        for (int k = 0; k < E / 8; ++k) {
          uint32_t ww[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            ww[e] = static_cast<uint32_t>(to_bf16_bits(v[8 * k + 2 * e])) |
                    (static_cast<uint32_t>(to_bf16_bits(v[8 * k + 2 * e + 1])) << 16);
          dst[k] = make_uint4(ww[0], ww[1], ww[2], ww[3]);
        }
      }
    }
    // the transform runs on every quad (its shuffles need whole warps); only history rows are stored
    // register stages: butterflies on pairs (c, c + hl) two at a time as float32 pairs
#pragma unroll
    for (int hl = 1; hl < E; hl <<= 1) {
#pragma unroll
      for (int c = 0; c < E; c += 2) {
        if (hl == 1) {
          if ((c & 1) == 0) {
            const float x0 = v[c], x1 = v[c + 1];
            v[c] = x0 + x1;
            v[c + 1] = x0 - x1;
          }
        } else if ((c & hl) == 0) {
          const float2 x0 = make_float2(v[c], v[c + 1]), x1 = make_float2(v[c + hl], v[c + hl + 1]);
          const float2 sm = __fadd2_rn(x0, x1), df = __fadd2_rn(x0, make_float2(-x1.x, -x1.y));
          v[c] = sm.x; v[c + 1] = sm.y;
          v[c + hl] = df.x; v[c + hl + 1] = df.y;
        }
      }
    }
    // quad stages: partner o; the lower lane keeps v + o, the upper o - v, as o + sign * v
#pragma unroll
    for (int lm = 1; lm < 4; lm <<= 1) {
      const float sgn = (q & lm) ? -1.f : 1.f;
#pragma unroll
      for (int c = 0; c < E; ++c) {
        const float o = __shfl_xor_sync(0xffffffffu, v[c], lm);
        v[c] = fmaf(sgn, v[c], o);
      }
    }
    const float inv_sqrt_d = D == 64 ? 0.125f : 0.08838834764831845f;  // 1/sqrt(D) rounded to float32
    uint8_t* crow = cbuf[warp][rl];
    const int bq = brev_bits(q, 2);
    uint32_t szw = 0;
#pragma unroll
    for (int cg = 0; cg < G; ++cg) {
      const int gi = brev_bits(cg, NG);
      // y = v / sqrt(D), rounded once; the group's extremes are found on v (rounding a
      // multiplication by a positive constant is monotonic) and then scaled
      float mn = v[cg], mx = v[cg];
#pragma unroll
      for (int m = 1; m < 8; ++m) {
        mn = fminf(mn, v[cg + G * m]);
        mx = fmaxf(mx, v[cg + G * m]);
      }
#pragma unroll
      for (int lm = 1; lm < 4; lm <<= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, lm));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, lm));
      }
      // clipping is monotonic: the clipped group's min and max are the clipped min and max
      mn = fminf(fmaxf(mn * inv_sqrt_d, -clip), clip);
      mx = fminf(fmaxf(mx * inv_sqrt_d, -clip), clip);
      const uint16_t zb = to_bf16_bits(mn);
      const uint16_t sb = to_bf16_bits((mx - mn) / 3.0f);
      const float z = __uint_as_float(static_cast<uint32_t>(zb) << 16);
      const float sc = __uint_as_float(static_cast<uint32_t>(sb) << 16);
      const float inv = sc > 0.f ? __frcp_rn(sc) : 0.f;  // s = 0: every code 0
      const float zinv = -z * inv;
      // code = clamp(rne((clip(y) - z) / s), 0, 3) as y * (1/s) - z/s clamped to the images of the
      // clip range and to [0, 3], rounded by adding 1.5 * 2^23 (the code is the pattern's low bits);
      // the image of clip is below 0 when the BF16 zero lands above a clip that BF16 cannot
      // represent and the group spans less than that rounding, so t_hi is kept at 0 or above
      const float t_lo = fmaxf(fmaf(-clip, inv, zinv), 0.f);
      const float t_hi = fmaxf(fminf(fmaf(clip, inv, zinv), 3.f), 0.f);
      uint32_t pat[8];
#pragma unroll
      for (int m = 0; m < 8; ++m)
        pat[m] = __float_as_uint(fminf(fmaxf(fmaf(v[cg + G * m] * inv_sqrt_d, inv, zinv), t_lo), t_hi) + 12582912.0f);
      // Channel u = 4 br3(m) + br2(q) of the group.  With mb = br3(m), the four codes of
      // mb = 2k + lo (k = 0..3) fill one byte of a page word, field k at bits 2k: the byte is
      // p0 + 4 p1 + 16 p2 + 64 p3 of the patterns (1.5 * 2^23 has a zero low byte).
#pragma unroll
      for (int lo = 0; lo < 2; ++lo) {
        uint32_t by = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) by += pat[brev_bits(2 * k + lo, 3)] << (2 * k);
        int w, bi;  // page word and byte within it
        if (!is_v) {
          w = (2 * lo + (bq >> 1)) * WPQ + (gi >> 1);
          bi = 2 * (bq & 1) + (gi & 1);
        } else {
          const int hw = WPQ * (4 * lo + bq) + (gi >> 1);
          w = hw >> 1;
          bi = 2 * (hw & 1) + (gi & 1);
        }
        crow[4 * w + bi] = static_cast<uint8_t>(by);
      }
      if (q == gi) szw = static_cast<uint32_t>(sb) | (static_cast<uint32_t>(zb) << 16);
    }
    __syncwarp();
    if (kind == 1) {
      if (page < 0 || page >= g.num_pages) {
        if (q == 0) flag_error(a.status, kDevBadPage);
      } else {
        uint8_t* codes;
        uint32_t* sz;
        history_row_ptrs<D>(a, page, t & (g.P - 1), h, is_v, &codes, &sz);
        if constexpr (WPQ == 2) reinterpret_cast<uint2*>(codes)[q] = reinterpret_cast<const uint2*>(crow)[q];
        else reinterpret_cast<uint32_t*>(codes)[q] = reinterpret_cast<const uint32_t*>(crow)[q];
        if (q < G) sz[q] = szw;
      }
    }
    __syncwarp();
  }
}

// ------------------------------------------------------------------ eviction before an extend
// Ring tokens [max(S, t0-W), min(t0, n1-W)) of request b become history.
// grid = (ceil(W / warps), batch, 2): one warp per (ring position, all heads).
template <int D>
__global__ void __launch_bounds__(kWarpsPerCta * 32) evict_kernel(WriteArgs a) {
  __shared__ WarpSmem sm[kWarpsPerCta];
  pdl_launch_dependents();  // the write kernel after it may start its set-up; it waits before its stores
  pdl_wait();               // (when launched as a programmatic dependent) everything before it is complete
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Geom& g = a.g;
  const int b = blockIdx.y;
  const bool is_v = blockIdx.z == 1;
  const float* R = is_v ? a.R_V : a.R_K;
  const int i = blockIdx.x * kWarpsPerCta + warp;
  const int t0 = a.start_pos[b];
  const int n1 = t0 + (a.cu_seqlens[b + 1] - a.cu_seqlens[b]);
  const int e0 = max(g.S, t0 - g.W);
  const int e1 = min(t0, n1 - g.W);
  const int e = e0 + i;
  if (i >= g.W || e >= e1) return;
  if (t0 < 0 || n1 > g.max_pages_per_req * g.P) {
    if (lane == 0) flag_error(a.status, kDevBadLen);
    return;
  }
  const int req = a.req_slot[b];
  if (req < 0 || req >= g.max_req) {
    if (lane == 0) flag_error(a.status, kDevBadSlot);
    return;
  }
  for (int h = 0; h < g.Hkv; ++h) {
    const uint16_t* ring = window_row(a, req, h, is_v, window_slot(e, g.S, g.W));
    for (int c = lane; c < D; c += 32) sm[warp].x[c] = __uint_as_float(static_cast<uint32_t>(ring[c]) << 16);
    __syncwarp();
    store_history<D>(a, b, e, h, is_v, sm[warp].x, R + (size_t)h * g.rot_stride(), sm[warp].codes, sm[warp].f);
    __syncwarp();
  }
}

// ------------------------------------------------------------------ decode append
// grid = (batch, 2, ceil(Hkv / kAppendHeads)), block = 4 warps, dynamic shared
// memory = one rotation (D*D floats).  blockIdx.y selects K (0) or V (1); the
// CTA handles kAppendHeads kv heads.  One bulk copy brings R_K or R_V into
// shared memory; warp k runs rotation chain k (input channels [kD/4, (k+1)D/4))
// for every head of the CTA, lane l producing outputs [lC, (l+1)C); the chains
// meet in shared memory and warp h adds them in the canonical order for head
// h, quantises and packs.  The CTA reads the evicted token's ring row before
// overwriting that slot with the new token.
constexpr int kAppendHeads = 2;

// kv heads served by one append CTA: kAppendHeads share the CTA's staged rotation, so with a
// rotation per kv head a CTA serves one head
__host__ __device__ inline int append_heads_per_cta(const Geom& g) { return g.rph ? 1 : kAppendHeads; }

// Returns false if the rotation copy timed out (flagged; nothing written).
// (b, by, bz): request, K|V, head group.  early_r: the fused step's form, which
// fetches R (a per-layer constant) first and then waits on the preceding grid
// before it reads anything that grid may write.
template <int D>
__device__ __forceinline__ bool append_body(const WriteArgs& a, float* Rsm, uint64_t* bar, int b, int by, int bz,
                                            bool early_r) {
  constexpr int C = D / 32;
  constexpr int HPC = kAppendHeads;
  __shared__ float xs[HPC][D];
  __shared__ float part[4][HPC][D];
  __shared__ uint8_t code_scratch[HPC][D];
  __shared__ uint16_t new_row[HPC][D];   // the new token, BF16
  __shared__ int page_sh;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Geom& g = a.g;
  const bool is_v = by == 1;
  const int hpc = append_heads_per_cta(g);
  const int h0 = bz * hpc;
  const int nh = min(hpc, g.Hkv - h0);
  const float* Rg = (is_v ? a.R_V : a.R_K) + (size_t)h0 * g.rot_stride();  // the rotation of this CTA's heads
  if (early_r) {
    if (threadIdx.x == 0) {
      mbar_init(bar, 1);
      fence_barrier_init();
      mbar_arrive_expect_tx(bar, D * D * sizeof(float));
      bulk_g2s(Rsm, Rg, D * D * sizeof(float), bar);
    }
    pdl_wait();
  }
  // an exit that leaves the early rotation copy unused waits for it first
  auto drain = [&]() {
    if (early_r && threadIdx.x == 0) (void)mbar_wait_bounded(bar, 0, nullptr);
  };
  const int n0 = a.start_pos[b] + a.start_offset;
  if (n0 < 0 || n0 + 1 > g.max_pages_per_req * g.P) {
    if (threadIdx.x == 0) flag_error(a.status, kDevBadLen);
    drain();
    return true;
  }
  const int req = a.req_slot[b];
  if (req < 0 || req >= g.max_req) {
    if (threadIdx.x == 0) flag_error(a.status, kDevBadSlot);
    drain();
    return true;
  }
  const int slot_new = window_slot(n0, g.S, g.W);
  const int e = n0 - g.W;
  const bool evict = e >= g.S;  // the evicted token occupies the slot the new token takes
  // every global read of this kernel happens before the dependent kernel is let
  // in: its page stream would otherwise queue ahead of them
  if (!early_r && evict && threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
    mbar_arrive_expect_tx(bar, D * D * sizeof(float));
    bulk_g2s(Rsm, Rg, D * D * sizeof(float), bar);
  }
  // issue the loads, let the dependent kernel launch (its first requests then
  // queue behind these), then consume them
  constexpr int PER = (HPC * D + 127) / 128;  // elements per thread (blockDim 128)
  const void* src = is_v ? a.V : a.K;
  float nv[PER], rv[PER];
  int pid = -1;
  if (evict && threadIdx.x == 32) {
    const int lp = e / g.P;
    if (lp < a.bt_stride && lp < g.max_pages_per_req) pid = a.block_table[(size_t)b * a.bt_stride + lp];
  }
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int idx = threadIdx.x + u * 128;
    nv[u] = rv[u] = 0.f;
    if (idx < nh * D) {
      const int hh = idx / D, c = idx % D;
      nv[u] = load_in(src, a.dtype, ((size_t)b * g.Hkv + h0 + hh) * D + c);
      if (evict) rv[u] = __uint_as_float(static_cast<uint32_t>(window_row(a, req, h0 + hh, is_v, slot_new)[c]) << 16);
    }
  }
  pdl_launch_dependents();
#pragma unroll
  for (int u = 0; u < PER; ++u) {
    const int idx = threadIdx.x + u * 128;
    if (idx < nh * D) {
      new_row[idx / D][idx % D] = to_bf16_bits(nv[u]);
      xs[idx / D][idx % D] = rv[u];
    }
  }
  if (evict && threadIdx.x == 32) {
    if (pid < 0 || pid >= g.num_pages) {
      flag_error(a.status, kDevBadPage);
      pid = -1;
    }
    page_sh = pid;
  }
  __syncthreads();
  if (evict && !mbar_wait_bounded(bar, 0, a.status)) {
    (void)mbar_wait_bounded(bar, 0, nullptr);
    return false;  // uniform: every thread times out on the same copy
  }
  if (!evict) drain();
  if (evict) {
    float acc[HPC][C];
#pragma unroll
    for (int hh = 0; hh < HPC; ++hh)
#pragma unroll
      for (int c = 0; c < C; ++c) acc[hh][c] = 0.f;
#pragma unroll 8
    for (int i = 0; i < D / 4; ++i) {
      const int ii = warp * (D / 4) + i;
      const float* r = Rsm + ii * D + lane * C;
#pragma unroll
      for (int hh = 0; hh < HPC; ++hh) {
        const float xi = xs[hh][ii];
#pragma unroll
        for (int c = 0; c < C; ++c) acc[hh][c] = fmaf(xi, r[c], acc[hh][c]);
      }
    }
#pragma unroll
    for (int hh = 0; hh < HPC; ++hh)
#pragma unroll
      for (int c = 0; c < C; ++c) part[warp][hh][lane * C + c] = acc[hh][c];
  }
  __syncthreads();
  if (evict && warp < nh) {
    float y[C];
#pragma unroll
    for (int c = 0; c < C; ++c) {
      const int j = lane * C + c;
      y[c] = ((part[0][warp][j] + part[1][warp][j]) + part[2][warp][j]) + part[3][warp][j];
    }
    const int page = page_sh;
    if (page >= 0) {
      uint8_t* codes;
      uint32_t* sz;
      history_row_ptrs<D>(a, page, e % g.P, h0 + warp, is_v, &codes, &sz);
      quant_pack_store<D>(y, is_v ? a.clip_V : a.clip_K, is_v, codes, sz, code_scratch[warp]);
    }
  }
  // the new token takes the ring slot (the evicted row was read above)
  for (int idx = threadIdx.x; idx < nh * D; idx += blockDim.x) {
    const int hh = idx / D, c = idx % D;
    window_row(a, req, h0 + hh, is_v, slot_new)[c] = new_row[hh][c];
  }
  return true;
}

// Launched after the query rotation of a fused decode step (programmatic
// dependent launch), the append runs alongside it.  It lets the split-K kernel
// launch once its own reads are issued, and waits for its predecessor only at
// the end, so that its completion implies the rotation's.  Launched on its
// own, both are no-ops.
template <int D>
__global__ void __launch_bounds__(128) append_kernel(WriteArgs a) {
  extern __shared__ __align__(16) float Rsm[];  // [D][D]
  __shared__ __align__(8) uint64_t bar;
  (void)append_body<D>(a, Rsm, &bar, blockIdx.x, blockIdx.y, blockIdx.z, false);
  pdl_launch_dependents();  // no-op if already done; covers the early exits
  pdl_wait();
}

// The first kernel of a fused decode step: CTAs [0, nq) rotate the query
// (q_rotate_cta, nq = Hkv * D/32 * batch; none when the decode is one launch,
// whose split CTAs form the query side), the rest run the append, one grid
// instead of two so that no second launch sits on the step's critical path.
// Every CTA waits on the preceding grid before it reads anything that grid may
// write; the split-K kernel, its programmatic dependent, waits for the whole grid.
template <int D>
__global__ void __launch_bounds__(128) step_prep_kernel(const __grid_constant__ WriteArgs w,
                                                        const __grid_constant__ DecodeArgs d) {
  extern __shared__ __align__(16) float Rsm[];  // [D][D] (append) or the rotation's arrays
  __shared__ __align__(8) uint64_t bar;
  const int qx = d.g.Hkv * (D / 32);
  const int nq = d.wl.fused ? 0 : qx * d.batch;
  if ((int)blockIdx.x < nq) {
    q_rotate_cta<D>(d, blockIdx.x % (D / 32), (blockIdx.x % qx) / (D / 32), blockIdx.x / qx, Rsm,
                    q_out_ws(d, (blockIdx.x % qx) / (D / 32), blockIdx.x / qx));
    return;
  }
  const int i = blockIdx.x - nq;
  const int nz = (w.g.Hkv + append_heads_per_cta(w.g) - 1) / append_heads_per_cta(w.g);
  (void)append_body<D>(w, Rsm, &bar, i / (2 * nz), (i % (2 * nz)) / nz, (i % (2 * nz)) % nz, true);
  pdl_launch_dependents();  // covers the early exits
}

}  // namespace

template <int D>
int launch_write_t(const WriteArgs& a, cudaStream_t s, bool pdl) {
  const int heads = a.g.rph ? a.g.Hkv : 1;  // grid z: one kv head per z with a rotation per kv head
  const long long rows = (long long)a.total_tokens * a.g.Hkv / heads;
  long long ctas = (rows + kWarpsPerCta * kRowsPerPass - 1) / (kWarpsPerCta * kRowsPerPass);
  if (ctas * heads > 152 * 2) ctas = (152 * 2 + heads - 1) / heads;  // two CTAs per SM fit (R + row buffers)
  const size_t smem = sizeof(float) * D * D + sizeof(WriteSmem<D>);
  cudaError_t e = ensure_smem_limit(write_kernel<D>, smem);
  if (e != cudaSuccess) return (int)e;
  return launch_pdl(write_kernel<D>, dim3((unsigned)ctas, 2, (unsigned)heads), dim3(kWarpsPerCta * 32), smem, s, pdl, a);
}

template <int D>
int launch_write_fwht_t(const WriteArgs& a, cudaStream_t s, bool pdl) {
  const long long rows = (long long)a.total_tokens * a.g.Hkv;
  long long ctas = (rows + kFwhtWarps * 8 - 1) / (kFwhtWarps * 8);
  // one wave (K and V CTAs together fill the SMs at the kernel's occupancy), then a grid-stride loop
  static int per_sm = 0;
  if (per_sm == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, write_fwht_kernel<D>, kFwhtWarps * 32, 0) != cudaSuccess ||
        n < 1)
      n = 1;
    per_sm = n;
  }
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms < 1)
    sms = 152;
  const long long cap = (long long)sms * per_sm / 2 > 0 ? (long long)sms * per_sm / 2 : 1;
  if (ctas > cap) ctas = cap;
  return launch_pdl(write_fwht_kernel<D>, dim3((unsigned)ctas, 2), dim3(kFwhtWarps * 32), 0, s, pdl, a);
}

int launch_write(const WriteArgs& a, void* stream, bool pdl) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long rows = (long long)a.total_tokens * a.g.Hkv;
  if (rows == 0) return 0;
  // the quad-lane transform reads each quarter row with 16-byte loads
  const bool aligned = ((reinterpret_cast<uintptr_t>(a.K) | reinterpret_cast<uintptr_t>(a.V)) & 15) == 0;
  if (a.hadamard && aligned)
    return a.g.D == 128 ? launch_write_fwht_t<128>(a, s, pdl) : launch_write_fwht_t<64>(a, s, pdl);
  return a.g.D == 128 ? launch_write_t<128>(a, s, pdl) : launch_write_t<64>(a, s, pdl);
}

int launch_evict(const WriteArgs& a, void* stream, bool pdl) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (a.batch == 0) return 0;
  dim3 grid((a.g.W + kWarpsPerCta - 1) / kWarpsPerCta, a.batch, 2);
  if (a.g.D == 128) return launch_pdl(evict_kernel<128>, grid, dim3(kWarpsPerCta * 32), 0, s, pdl, a);
  return launch_pdl(evict_kernel<64>, grid, dim3(kWarpsPerCta * 32), 0, s, pdl, a);
}

int launch_step_prep(const WriteArgs& w, const DecodeArgs& d, void* stream, bool pdl) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (w.batch == 0) return 0;
  const int nz = (w.g.Hkv + append_heads_per_cta(w.g) - 1) / append_heads_per_cta(w.g);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((d.wl.fused ? 0 : d.g.Hkv * (d.g.D / 32) * d.batch) + w.batch * 2 * nz);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = sizeof(float) * w.g.D * w.g.D;   // holds the rotation's arrays as well
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  auto go = [&](auto kern) -> int {
    cudaError_t e = ensure_smem_limit(kern, cfg.dynamicSmemBytes);
    if (e != cudaSuccess) return (int)e;
    return (int)cudaLaunchKernelEx(&cfg, kern, w, d);
  };
  return w.g.D == 128 ? go(step_prep_kernel<128>) : go(step_prep_kernel<64>);
}

int launch_append(const WriteArgs& a, void* stream, bool pdl) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (a.batch == 0) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.batch, 2, (a.g.Hkv + append_heads_per_cta(a.g) - 1) / append_heads_per_cta(a.g));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = sizeof(float) * a.g.D * a.g.D;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  cudaError_t e;
  if (a.g.D == 128) {
    if ((e = ensure_smem_limit(append_kernel<128>, cfg.dynamicSmemBytes)) != cudaSuccess) return (int)e;
    return (int)cudaLaunchKernelEx(&cfg, append_kernel<128>, a);
  }
  if ((e = ensure_smem_limit(append_kernel<64>, cfg.dynamicSmemBytes)) != cudaSuccess) return (int)e;
  return (int)cudaLaunchKernelEx(&cfg, append_kernel<64>, a);
}

}  // namespace oscar
