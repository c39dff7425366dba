// In-house BF16 paged decode: the comparison point for the OSCAR claim that
// INT2 history makes batch-1 decode faster than BF16 by cutting KV memory
// traffic (arXiv abstract; gist.science summary, section 4).  Standard
// split-K flash decoding over an all-BF16 paged cache, written the same way as
// the INT2 kernel: one CTA per (split, kv head, request), 4 warps, a 3-stage
// shared-memory ring of whole pages, mma.sync m16n8k16 for QK and PV with the
// GQA heads as the N dimension, online softmax in the log2 domain, a combine
// kernel for the split partials.
//
// Pages are staged with TMA tensor copies (cp.async.bulk.tensor.2d, no
// multicast) in 128-byte swizzle so that ldmatrix reads of 256-byte rows are
// free of bank conflicts.  The pool is viewed as a 2-D tensor of bf16 rows:
// row ((((layer*num_pages + page)*Hkv + h)*2 + kv)*P + slot), D columns; one
// box is P rows x 64 columns (128 bytes).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "oscar_internal.h"

namespace oscar {
namespace {

constexpr int kThreads = 128;
constexpr int kStages = 3;
constexpr float kLog2e = 1.4426950408889634f;

struct WsView {
  uint2* qfrag;   // [B][Hkv][NT][D/16][32]
  float* part;    // [B][Hq][max_splits][D + 4]
};

__device__ __forceinline__ WsView ws_view(const DecodeArgs& a) {
  WsView v;
  v.qfrag = reinterpret_cast<uint2*>(a.ws + a.wl.qfrag_off);
  v.part = reinterpret_cast<float*>(a.ws + a.wl.part_off);
  return v;
}

__device__ __forceinline__ bool seq_len_ok(const DecodeArgs& a, int n) {
  return n >= 0 && n <= a.max_seq && n <= a.g.max_pages_per_req * a.g.P;
}

__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// Byte offset of (row r, 16-byte chunk c) inside a 128B-swizzled box of 128-byte rows.
__device__ __forceinline__ uint32_t swz(int r, int c) { return r * 128 + ((c ^ (r & 7)) << 4); }

// ------------------------------------------------------------------ query fragments
// grid (Hq, B), block 64: thread j < D/16*8 writes one lane's (b0, b1) of one k-tile.
template <int D>
__global__ void __launch_bounds__(64) bf16_prepare_kernel(DecodeArgs a) {
  pdl_launch_dependents();
  const Geom& g = a.g;
  const int h = blockIdx.x, b = blockIdx.y, j = threadIdx.x;
  const int gq = g.gq(), kvh = h / gq, hh = h % gq, nt = hh >> 2;
  if (j >= (D / 16) * 8) return;
  const int kk = j >> 3, sub = j & 7, hl = sub >> 2, tig = sub & 3;
  const int gid = 2 * (hh & 3) + hl, lane = gid * 4 + tig;
  const size_t qbase = ((size_t)b * g.Hq + h) * D;
  uint32_t regs[2];
#pragma unroll
  for (int hp = 0; hp < 2; ++hp) {
    const int ch = 16 * kk + 8 * hp + 2 * tig;
    float v[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      float x;
      if (a.q_dtype == kDtypeBF16) x = __uint_as_float(static_cast<uint32_t>(static_cast<const uint16_t*>(a.q)[qbase + ch + u]) << 16);
      else x = static_cast<const float*>(a.q)[qbase + ch + u];
      const float hi = __bfloat162float(__float2bfloat16_rn(x));
      v[u] = hl ? (x - hi) : hi;
    }
    regs[hp] = pack_bf162(v[0], v[1]);
  }
  WsView ws = ws_view(a);
  ws.qfrag[((((size_t)b * g.Hkv + kvh) * a.wl.nt + nt) * (D / 16) + kk) * 32 + lane] = make_uint2(regs[0], regs[1]);
}

// ------------------------------------------------------------------ split-K decode
template <int D, int NT>
__global__ void __launch_bounds__(kThreads) bf16_decode_kernel(const __grid_constant__ CUtensorMap tmap, DecodeArgs a) {
  constexpr int P = 64;
  constexpr int HALF = P * 128;            // one box: P rows x 128 bytes
  constexpr int NCH = D / 64;              // boxes per K (or V) row block
  constexpr int STAGE = 2 * NCH * HALF;    // K and V of one page
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * STAGE);

  const Geom& g = a.g;
  const int b = blockIdx.z, kvh = blockIdx.y, split = blockIdx.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int gq = g.gq();
  const int n = a.seq_lens[b];
  if (!seq_len_ok(a, n)) {
    if (tid == 0 && split == 0) flag_error(a.status, kDevBadLen);
    pdl_launch_dependents();
    return;
  }
  const int n_pages = n > 0 ? (n - 1) / P + 1 : 0;
  const int pg0 = split * a.wl.pages_per_split;
  if (pg0 >= n_pages) { pdl_launch_dependents(); return; }
  const int pg1 = min(pg0 + a.wl.pages_per_split, n_pages);
  const int n_iters = pg1 - pg0;
  const int* bt = a.block_table + (size_t)b * a.bt_stride;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncthreads();
  __shared__ int stage_ok[kStages];
  auto issue = [&](int it) {
    const int s = it % kStages;
    const int lp = pg0 + it;
    const int pid = (lp < a.bt_stride && lp < g.max_pages_per_req) ? bt[lp] : -1;
    const bool ok = pid >= 0 && pid < g.num_pages;
    stage_ok[s] = ok;
    if (!ok) flag_error(a.status, kDevBadPage);
    mbar_arrive_expect_tx(&bars[s], ok ? STAGE : 0);
    if (ok) {
      const int row0 = ((((a.layer * g.num_pages + pid) * g.Hkv + kvh) * 2) * P);
#pragma unroll
      for (int kv = 0; kv < 2; ++kv)
#pragma unroll
        for (int c = 0; c < NCH; ++c)
          tma_load_2d(smem + s * STAGE + (kv * NCH + c) * HALF, &tmap, c * 64, row0 + kv * P, &bars[s]);
    }
  };
  if (tid == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap)) : "memory");
    for (int it = 0; it < kStages && it < n_iters; ++it) issue(it);
  }
  pdl_wait();
  WsView ws = ws_view(a);
  uint32_t qb[NT][D / 16][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const bool col_ok = (nt * 4 + (gid >> 1)) < gq;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint2 f = ws.qfrag[((((size_t)b * g.Hkv + kvh) * NT + nt) * (D / 16) + kk) * 32 + lane];
      qb[nt][kk][0] = col_ok ? f.x : 0u;
      qb[nt][kk][1] = col_ok ? f.y : 0u;
    }
  }
  const float sm_log2 = kLog2e * rsqrtf((float)D);
  float m_run[NT], l_run[NT], acc[NT][D / 16][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt] = -INFINITY;
    l_run[nt] = 0.f;
#pragma unroll
    for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[nt][mt][r] = 0.f;
  }
  const int r_base = 16 * warp;  // this warp's 16 token rows inside the page
  const int mrow = lane & 7, mat = lane >> 3;
  bool aborted = false;
  int it_fail = 0;
  for (int it = 0; it < n_iters; ++it) {
    const int s = it % kStages;
    const bool ok = mbar_wait_bounded(&bars[s], (it / kStages) & 1, a.status);
    if (ok) {
      const bool page_ok = stage_ok[s];
      const uint8_t* kbase = smem + s * STAGE;
      const uint8_t* vbase = kbase + NCH * HALF;
      const int t0 = (pg0 + it) * P + r_base;
      // QK: A = K rows (16 tokens x 16 channels) via ldmatrix; matrices (rows 0-7|8-15) x (k 0-7|8-15)
      float sc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int r = 0; r < 4; ++r) sc[nt][r] = 0.f;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int row = r_base + mrow + 8 * (mat & 1);
        const int chunk = (kk * 2 + (mat >> 1));          // 16-byte chunk along D
        const int box = chunk >> 3, cin = chunk & 7;
        uint32_t af[4];
        ldmatrix_x4(af, smem_u32(kbase + box * HALF + swz(row, cin)));
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma_bf16(sc[nt], af[0], af[1], af[2], af[3], qb[nt][kk][0], qb[nt][kk][1]);
      }
      const int ta = t0 + gid, tb = t0 + gid + 8;
      const bool va = page_ok && ta < n, vb = page_ok && tb < n;
      float pa[NT], pb[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float s_a = va ? (sc[nt][0] + sc[nt][1]) * sm_log2 : -INFINITY;
        const float s_b = vb ? (sc[nt][2] + sc[nt][3]) * sm_log2 : -INFINITY;
        float mb = fmaxf(s_a, s_b);
        mb = warp_max_xor(mb, 4);
        mb = warp_max_xor(mb, 8);
        mb = warp_max_xor(mb, 16);
        const float m_new = fmaxf(m_run[nt], mb);
        const float alpha = (m_new == -INFINITY) ? 1.f : ex2(m_run[nt] - m_new);
        pa[nt] = (s_a == -INFINITY) ? 0.f : ex2(s_a - m_new);
        pb[nt] = (s_b == -INFINITY) ? 0.f : ex2(s_b - m_new);
        m_run[nt] = m_new;
        l_run[nt] = fmaf(l_run[nt], alpha, pa[nt] + pb[nt]);
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt)
#pragma unroll
          for (int r = 0; r < 4; ++r) acc[nt][mt][r] *= alpha;
      }
      // PV: A = V^T (16 channels x 16 tokens) via ldmatrix.trans; B = p (tokens x (head, hi|lo))
      const int src0 = (2 * tig) * 4 + (gid >> 1), src1 = (2 * tig + 1) * 4 + (gid >> 1);
      const bool lo_lane = (gid & 1) != 0;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float pr[4] = {__shfl_sync(0xffffffffu, pa[nt], src0), __shfl_sync(0xffffffffu, pa[nt], src1),
                             __shfl_sync(0xffffffffu, pb[nt], src0), __shfl_sync(0xffffffffu, pb[nt], src1)};
        float wv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float hi = __bfloat162float(__float2bfloat16_rn(pr[u]));
          wv[u] = lo_lane ? (pr[u] - hi) : hi;
        }
        const uint32_t b0 = pack_bf162(wv[0], wv[1]), b1 = pack_bf162(wv[2], wv[3]);
#pragma unroll
        for (int mt = 0; mt < D / 16; ++mt) {
          // matrices: (tokens 0-7 | 8-15) x (channels 16mt+0..7 | 16mt+8..15)
          const int row = r_base + mrow + 8 * (mat >> 1);
          const int chunk = 2 * mt + (mat & 1);
          const int box = chunk >> 3, cin = chunk & 7;
          uint32_t vf[4];
          ldmatrix_x4_trans(vf, smem_u32(vbase + box * HALF + swz(row, cin)));
          mma_bf16(acc[nt][mt], vf[0], vf[1], vf[2], vf[3], b0, b1);
        }
      }
    }
    aborted = __syncthreads_or(!ok) != 0;
    if (aborted) { it_fail = it; break; }
    if (tid == 0 && it + kStages < n_iters) issue(it + kStages);
  }
  if (aborted) {
    if (tid == 0) {
      const int last = min(n_iters, it_fail + kStages);
      for (int it = it_fail; it < last; ++it) (void)mbar_wait_bounded(&bars[it % kStages], (it / kStages) & 1, nullptr);
    }
    __syncthreads();
    pdl_launch_dependents();
    return;
  }
  pdl_launch_dependents();
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    l_run[nt] += __shfl_xor_sync(0xffffffffu, l_run[nt], 4);
    l_run[nt] += __shfl_xor_sync(0xffffffffu, l_run[nt], 8);
    l_run[nt] += __shfl_xor_sync(0xffffffffu, l_run[nt], 16);
  }
  float* wm = reinterpret_cast<float*>(smem);
  float* wl = wm + 32;
  float* wacc = wl + 32;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int hh = nt * 4 + tig;
    if (hh < gq) {
      if (gid == 0) {
        wm[warp * 8 + hh] = m_run[nt];
        wl[warp * 8 + hh] = l_run[nt];
      }
#pragma unroll
      for (int mt = 0; mt < D / 16; ++mt) {
        wacc[(warp * 8 + hh) * D + 16 * mt + gid] = acc[nt][mt][0] + acc[nt][mt][1];
        wacc[(warp * 8 + hh) * D + 16 * mt + 8 + gid] = acc[nt][mt][2] + acc[nt][mt][3];
      }
    }
  }
  __syncthreads();
  for (int idx = tid; idx < gq * D; idx += kThreads) {
    const int hh = idx / D, ch = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, wm[w * 8 + hh]);
    float accv = 0.f, L = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float mw = wm[w * 8 + hh];
      const float f = (mw == -INFINITY) ? 0.f : ex2(mw - M);
      accv = fmaf(f, wacc[(w * 8 + hh) * D + ch], accv);
      L = fmaf(f, wl[w * 8 + hh], L);
    }
    float* pp = ws.part + (((size_t)b * g.Hq + kvh * gq + hh) * a.wl.max_splits + split) * (D + 4);
    pp[4 + ch] = accv;
    if (ch == 0) {
      pp[0] = M;
      pp[1] = L;
    }
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads) bf16_combine_kernel(DecodeArgs a) {
  pdl_wait();
  const Geom& g = a.g;
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x, lane = tid & 31;
  __shared__ float wts[1024];
  __shared__ float s_l;
  WsView ws = ws_view(a);
  const int n = a.seq_lens[b];
  const int n_pages = (seq_len_ok(a, n) && n > 0) ? (n - 1) / g.P + 1 : 0;
  const int nsp = min((n_pages + a.wl.pages_per_split - 1) / a.wl.pages_per_split, 1024);
  const float* base = ws.part + ((size_t)b * g.Hq + h) * a.wl.max_splits * (D + 4);
  if (tid < 32) {
    float M = -INFINITY;
    for (int i = lane; i < nsp; i += 32) M = fmaxf(M, base[(size_t)i * (D + 4)]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    for (int i = lane; i < nsp; i += 32) {
      const float mi = base[(size_t)i * (D + 4)];
      const float w = (mi == -INFINITY) ? 0.f : ex2(mi - M);
      wts[i] = w;
      L = fmaf(w, base[(size_t)i * (D + 4) + 1], L);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (lane == 0) s_l = L;
  }
  __syncthreads();
  if (tid < D) {
    float r = 0.f;
    for (int i = 0; i < nsp; ++i) r = fmaf(wts[i], base[(size_t)i * (D + 4) + 4 + tid], r);
    const float o = s_l > 0.f ? r / s_l : 0.f;
    const size_t oi = ((size_t)b * g.Hq + h) * D + tid;
    if (a.out_dtype == kDtypeBF16) {
      __nv_bfloat16 hb = __float2bfloat16_rn(o);
      static_cast<uint16_t*>(a.out)[oi] = *reinterpret_cast<uint16_t*>(&hb);
    } else {
      static_cast<float*>(a.out)[oi] = o;
    }
  }
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
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

template <int D, int NT>
int launch_bf16_t(const DecodeArgs& a, cudaStream_t s, bool pdl) {
  constexpr int P = 64;
  constexpr int STAGE = 2 * (D / 64) * P * 128;
  auto enc = get_encode();
  if (!enc) return (int)cudaErrorNotSupported;
  CUtensorMap map;
  const uint64_t rows = (uint64_t)a.g.L * a.g.num_pages * a.g.Hkv * 2 * P;
  cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)D * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)P};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint8_t*>(a.bf16_pool), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return (int)cudaErrorInvalidValue;
  const size_t smem = kStages * STAGE + 1024 + kStages * 8;
  auto kern = bf16_decode_kernel<D, NT>;
  cudaError_t e = ensure_smem_limit(kern, smem);
  if (e != cudaSuccess) return (int)e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.wl.max_splits, a.g.Hkv, a.batch);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return (int)cudaLaunchKernelEx(&cfg, kern, map, a);
}

}  // namespace

int launch_bf16_prepare(const DecodeArgs& a, void* stream) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  dim3 grid(a.g.Hq, a.batch);
  if (a.g.D == 128) bf16_prepare_kernel<128><<<grid, 64, 0, s>>>(a);
  else bf16_prepare_kernel<64><<<grid, 64, 0, s>>>(a);
  return (int)cudaGetLastError();
}

int launch_bf16_decode(const DecodeArgs& a, void* stream, bool pdl) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (a.g.P != 64) return (int)cudaErrorNotSupported;
  if (a.wl.max_splits == 0) return 0;
  const int nt = a.wl.nt;
  if (a.g.D == 128) return nt == 2 ? launch_bf16_t<128, 2>(a, s, pdl) : launch_bf16_t<128, 1>(a, s, pdl);
  return nt == 2 ? launch_bf16_t<64, 2>(a, s, pdl) : launch_bf16_t<64, 1>(a, s, pdl);
}

int launch_bf16_combine(const DecodeArgs& a, void* stream, bool pdl) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.g.Hq, a.batch);
  cfg.blockDim = dim3(kThreads);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (a.g.D == 128) return (int)cudaLaunchKernelEx(&cfg, bf16_combine_kernel<128>, a);
  return (int)cudaLaunchKernelEx(&cfg, bf16_combine_kernel<64>, a);
}

}  // namespace oscar
