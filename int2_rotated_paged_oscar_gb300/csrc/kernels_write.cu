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
// One warp handles one (token, kv head, K|V) row: lane l owns channels
// [l*D/32, (l+1)*D/32).  The rotation y_j = sum_i x_i R[i][j] runs in float32
// with one FMA per term in increasing i, the same order in every kernel of this
// file, so the append, eviction and prefill paths produce identical codes for
// the same BF16 input.  The Hadamard-only variant replaces the dense product by
// a fast Walsh-Hadamard transform followed by the bit-reversal gather.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "oscar_internal.h"

namespace oscar {
namespace {

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
#pragma unroll
    for (int c = 0; c < C; ++c) y[c] = 0.f;
#pragma unroll 4
    for (int i = 0; i < D; ++i) {
      const float xi = xs[i];
      const float* r = R + (size_t)i * D + lane * C;
#pragma unroll
      for (int c = 0; c < C; ++c) y[c] = fmaf(xi, r[c], y[c]);
    }
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
// grid.x covers total_tokens * Hkv rows for one of K (blockIdx.y = 0) or V (1).
template <int D>
__global__ void __launch_bounds__(kWarpsPerCta * 32) write_kernel(WriteArgs a) {
  __shared__ WarpSmem sm[kWarpsPerCta];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool is_v = blockIdx.y == 1;
  const Geom& g = a.g;
  const void* src = is_v ? a.V : a.K;
  const float* R = is_v ? a.R_V : a.R_K;
  const long long rows = (long long)a.total_tokens * g.Hkv;
  for (long long item = (long long)blockIdx.x * kWarpsPerCta + warp; item < rows;
       item += (long long)gridDim.x * kWarpsPerCta) {
    const int row = static_cast<int>(item / g.Hkv);
    const int h = static_cast<int>(item % g.Hkv);
    // request of this row: largest b with cu_seqlens[b] <= row
    int lo = 0, hi = a.batch - 1;
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
      for (int i = lane; i < D; i += 32) sm[warp].x[i] = load_in(src, a.dtype, in_base + i);
      __syncwarp();
      store_history<D>(a, b, t, h, is_v, sm[warp].x, R, sm[warp].codes, sm[warp].f);
      __syncwarp();
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
}

// ------------------------------------------------------------------ eviction before an extend
// Ring tokens [max(S, t0-W), min(t0, n1-W)) of request b become history.
// grid = (ceil(W / warps), batch, 2): one warp per (ring position, all heads).
template <int D>
__global__ void __launch_bounds__(kWarpsPerCta * 32) evict_kernel(WriteArgs a) {
  __shared__ WarpSmem sm[kWarpsPerCta];
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
    store_history<D>(a, b, e, h, is_v, sm[warp].x, R, sm[warp].codes, sm[warp].f);
    __syncwarp();
  }
}

// ------------------------------------------------------------------ decode append
// grid = (batch, Hkv), block = 2 warps (K, V).
template <int D>
__global__ void __launch_bounds__(64) append_kernel(WriteArgs a) {
  __shared__ WarpSmem sm[2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Geom& g = a.g;
  const int b = blockIdx.x, h = blockIdx.y;
  const bool is_v = warp == 1;
  const float* R = is_v ? a.R_V : a.R_K;
  const int n0 = a.start_pos[b];
  if (n0 < 0 || n0 + 1 > g.max_pages_per_req * g.P) {
    if (lane == 0) flag_error(a.status, kDevBadLen);
    return;
  }
  const int req = a.req_slot[b];
  if (req < 0 || req >= g.max_req) {
    if (lane == 0) flag_error(a.status, kDevBadSlot);
    return;
  }
  const int slot_new = window_slot(n0, g.S, g.W);
  uint16_t* ring = window_row(a, req, h, is_v, slot_new);
  const int e = n0 - g.W;
  if (e >= g.S) {
    // the evicted token occupies the slot the new token takes
    for (int c = lane; c < D; c += 32) sm[warp].x[c] = __uint_as_float(static_cast<uint32_t>(ring[c]) << 16);
    __syncwarp();
    store_history<D>(a, b, e, h, is_v, sm[warp].x, R, sm[warp].codes, sm[warp].f);
    __syncwarp();
  }
  const void* src = is_v ? a.V : a.K;
  const size_t in_base = ((size_t)b * g.Hkv + h) * D;
  for (int c = lane; c < D; c += 32) ring[c] = to_bf16_bits(load_in(src, a.dtype, in_base + c));
}

int grid_for_rows(long long rows) {
  long long ctas = (rows + kWarpsPerCta - 1) / kWarpsPerCta;
  if (ctas > 152 * 16) ctas = 152 * 16;
  if (ctas < 1) ctas = 1;
  return static_cast<int>(ctas);
}

}  // namespace

int launch_write(const WriteArgs& a, void* stream) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long rows = (long long)a.total_tokens * a.g.Hkv;
  if (rows == 0) return 0;
  dim3 grid(grid_for_rows(rows), 2);
  if (a.g.D == 128) write_kernel<128><<<grid, kWarpsPerCta * 32, 0, s>>>(a);
  else write_kernel<64><<<grid, kWarpsPerCta * 32, 0, s>>>(a);
  return static_cast<int>(cudaGetLastError());
}

int launch_evict(const WriteArgs& a, void* stream) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (a.batch == 0) return 0;
  dim3 grid((a.g.W + kWarpsPerCta - 1) / kWarpsPerCta, a.batch, 2);
  if (a.g.D == 128) evict_kernel<128><<<grid, kWarpsPerCta * 32, 0, s>>>(a);
  else evict_kernel<64><<<grid, kWarpsPerCta * 32, 0, s>>>(a);
  return static_cast<int>(cudaGetLastError());
}

int launch_append(const WriteArgs& a, void* stream) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (a.batch == 0) return 0;
  dim3 grid(a.batch, a.g.Hkv);
  if (a.g.D == 128) append_kernel<128><<<grid, 64, 0, s>>>(a);
  else append_kernel<64><<<grid, 64, 0, s>>>(a);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace oscar
