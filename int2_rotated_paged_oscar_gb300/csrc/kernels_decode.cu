// Fused decode attention over the mixed-precision paged cache (INT2 history +
// BF16 sink/recent window).
//
// Source: OSCAR technical summary (gist.science), section 2.2 B -- the serving
// kernel unpacks, dequantises and inverse-rotates the INT2 history and computes
// attention over it, compatible with paged attention and prefix caching, with
// no extra memory traffic; arXiv abstract -- fused decode kernel, batch-1
// decode faster than BF16 by cutting KV memory traffic.
//
// Formulation (exact rearrangement of softmax(q K^T/sqrt(d)) V over
// K = [Y_K R_K^T ; K_win], V = [Y_V R_V^T ; V_win]):
//   q' = q R_K once per step;  history score_t = q'.y_K,t / sqrt(d);
//   history values accumulate in the rotated basis, acc_rot = sum_t p_t y_V,t;
//   o = (sum_win p v + acc_rot R_V^T) / l, R_V^T applied once per output row.
//
// Kernels (one decode step):
//   q_rotate       q' = q R_K per (request, q head); writes the query-side MMA
//                  fragments (f16 hi/lo split, per-head power-of-two scale),
//                  the group sums Q_g = sum_{j in g} q'_j, and q as float32.
//   decode_splitk  grid (1 + splits, kv heads, requests).  x = 0 is the BF16
//                  window split (CUDA cores, float32); x >= 1 streams a range of
//                  INT2 pages through a 4-stage shared-memory ring filled by
//                  non-multicast bulk copies (one per (page, kv head) block,
//                  mbarrier completion), and runs QK and PV on the tensor cores
//                  with mma.sync m16n8k16:
//                    QK  M = 16 tokens, N = (q head, f16 hi|lo), K = 16 channels,
//                        A = K codes unpacked to c*2^(pos-10) in f16 (exact),
//                        B = q' * 2^(e_h) * 2^(10-pos) split hi/lo; one
//                        accumulator per 32-channel group so the BF16 scale and
//                        zero apply in the float32 epilogue;
//                    PV  M = 16 channels, N = (q head, bf16 hi|lo), K = 16 tokens,
//                        A = V codes unpacked to c*2^(pos-7) in bf16 (exact),
//                        B = p_t * scale_{t,g} split hi/lo; the zero term
//                        sum_t p_t zero_{t,g} accumulates in float32.
//                  Online softmax in the log2 domain with float32 max/sum.
//   decode_combine merges the split partials, applies R_V^T once and divides by l.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <mutex>

#include "common.cuh"
#include "oscar_internal.h"

namespace oscar {

// Scratch of the allocation-free decode entry point (oscar_decode_attn_noalloc):
// a file-scope device array of kStaticScratchBytes.  Every GPU that loads the
// library holds it until the process exits.  Host code never uses the symbol
// as an address; it asks the runtime for the device address once per device
// (static_decode_scratch below).
static __device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

namespace {

constexpr int kThreads = 128;  // 4 warps
constexpr int kStages = 4;
constexpr int kStageTokens = 64;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxSplits = 1023;  // the host plan never asks for more

// ------------------------------------------------------------------ workspace views
struct WsView {
  uint2* qfrag;   // [B][Hkv][NT][D/16][32]
  float* qaux;    // [B][Hq][8]: [0] = 2^-e_h, [1 + g] = Q_g
  float* qplain;  // [B][Hq][D]
  float* part;    // [B][Hq][max_splits + 1][D + 4]: [0] m (log2 domain), [1] l, [4..] acc
};

__device__ __forceinline__ WsView ws_view(const DecodeArgs& a) {
  WsView v;
  v.qfrag = reinterpret_cast<uint2*>(a.ws + a.wl.qfrag_off);
  v.qaux = reinterpret_cast<float*>(a.ws + a.wl.qaux_off);
  v.qplain = reinterpret_cast<float*>(a.ws + a.wl.qplain_off);
  v.part = reinterpret_cast<float*>(a.ws + a.wl.part_off);
  return v;
}

__device__ __forceinline__ float load_q(const DecodeArgs& a, size_t idx) {
  if (a.q_dtype == kDtypeBF16) {
    const uint16_t v = static_cast<const uint16_t*>(a.q)[idx];
    return __uint_as_float(static_cast<uint32_t>(v) << 16);
  }
  return static_cast<const float*>(a.q)[idx];
}

// Number of INT2 splits request b needs (0 if it has no history).
__device__ __forceinline__ int splits_for(const DecodeArgs& a, int n) {
  const int h_end = n - a.g.W;
  if (h_end <= a.g.S) return 0;
  const int pages = (h_end - 1) / a.g.P + 1;
  return (pages + a.wl.pages_per_split - 1) / a.wl.pages_per_split;
}

__device__ __forceinline__ bool seq_len_ok(const DecodeArgs& a, int n) {
  return n >= 0 && n <= a.max_seq && n <= a.g.max_pages_per_req * a.g.P;
}

// ------------------------------------------------------------------ q rotate
// grid (Hq, B), block 128.  Thread j < D computes q'_j = sum_i q_i R_K[i][j].
template <int D>
__global__ void __launch_bounds__(kThreads) q_rotate_kernel(DecodeArgs a) {
  pdl_launch_dependents();
  const Geom& g = a.g;
  const int h = blockIdx.x, b = blockIdx.y;
  const int j = threadIdx.x;
  const int gq = g.gq();
  const int kvh = h / gq, hh = h % gq;
  const int nt = hh >> 2;
  __shared__ float qs[D];
  __shared__ float qr[D];
  __shared__ float red[kThreads / 32];
  WsView ws = ws_view(a);
  const size_t qbase = ((size_t)b * g.Hq + h) * D;
  if (j < D) {
    qs[j] = load_q(a, qbase + j);
    ws.qplain[qbase + j] = qs[j];
  }
  __syncthreads();
  float acc = 0.f;
  if (j < D) {
    for (int i = 0; i < D; ++i) acc = fmaf(qs[i], a.R_K[(size_t)i * D + j], acc);
    qr[j] = acc;
  }
  float m = j < D ? fabsf(acc) : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  // group sums: group gi = channels [32 gi, 32 gi + 32) = warp gi
  float gs = j < D ? acc : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) gs += __shfl_xor_sync(0xffffffffu, gs, o);
  if ((j & 31) == 0) red[j >> 5] = m;
  __syncthreads();
  float mx = 0.f;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) mx = fmaxf(mx, red[w]);
  int e = 0;
  if (mx > 0.f) {
    int E;
    frexpf(mx, &E);  // mx = f * 2^E, f in [0.5, 1)
    e = 5 - E;       // mx * 2^e in [16, 32): times 2^(10-pos) <= 1024 stays below the f16 maximum
  }
  float* aux = ws.qaux + ((size_t)b * g.Hq + h) * 8;
  if (j == 0) aux[0] = ldexpf(1.f, -e);
  if ((j & 31) == 0 && (j >> 5) < D / 32) aux[1 + (j >> 5)] = gs;
  // query-side fragments of the QK MMA: this head owns columns 2*(hh%4) + {hi, lo}
  if (j < (D / 16) * 8) {
    const int kk = j >> 3;  // k-tile = (group, kt)
    const int sub = j & 7;
    const int hl = sub >> 2, tig = sub & 3;
    const int gid = 2 * (hh & 3) + hl;
    const int lane = gid * 4 + tig;
    const int gi = kk >> 1, kt = kk & 1;
    const int p8 = 4 * gi + 2 * kt;
    uint32_t regs[2];
#pragma unroll
    for (int hpair = 0; hpair < 2; ++hpair) {
      const int ch = 32 * gi + 16 * kt + 8 * hpair + 2 * tig;
      const int pos = slot_pos((p8 + hpair) & 7);
      float v[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const float x = ldexpf(qr[ch + u], e + 10 - pos);
        const __half hi = __float2half_rn(x);
        const float lo = x - __half2float(hi);
        v[u] = hl ? lo : __half2float(hi);
      }
      regs[hpair] = pack_half2(v[0], v[1]);
    }
    const size_t fidx = ((((size_t)b * g.Hkv + kvh) * a.wl.nt + nt) * (D / 16) + kk) * 32 + lane;
    ws.qfrag[fidx] = make_uint2(regs[0], regs[1]);
  }
}

// ------------------------------------------------------------------ window split (BF16, float32 math)
template <int D, int NT>
__device__ void window_split(const DecodeArgs& a, int b, int kvh, float* smem_f) {
  const Geom& g = a.g;
  const int gq = g.gq();
  const int n = a.seq_lens[b];
  const int win = g.window();
  float* qsm = smem_f;                 // [gq][D]
  float* sc = qsm + 8 * D;             // [win][8]
  float* red = sc + win * 8;           // [4][8]
  WsView ws = ws_view(a);
  const int tid = threadIdx.x;
  for (int i = tid; i < gq * D; i += kThreads)
    qsm[i] = ws.qplain[((size_t)b * g.Hq + kvh * gq) * D + i];
  __syncthreads();
  const size_t sbase = ((size_t)a.layer * g.max_req + a.req_slot[b]) * g.slab_req_elems();
  const uint16_t* kwin = a.slab + sbase + ((size_t)kvh * 2 + 0) * win * D;
  const uint16_t* vwin = a.slab + sbase + ((size_t)kvh * 2 + 1) * win * D;
  const int n_recent = n > g.S ? min(n - g.S, g.W) : 0;
  const float sm = kLog2e * rsqrtf((float)D);
  for (int i = tid; i < win; i += kThreads) {
    const bool valid = i < g.S ? (i < n) : (i - g.S < n_recent);
    float acc[8];
#pragma unroll
    for (int hh = 0; hh < 8; ++hh) acc[hh] = 0.f;
    if (valid) {
      const uint32_t* kr = reinterpret_cast<const uint32_t*>(kwin + (size_t)i * D);
      for (int c2 = 0; c2 < D / 2; ++c2) {
        const uint32_t w = kr[c2];
        const float k0 = bf16_lo(w), k1 = bf16_hi(w);
#pragma unroll
        for (int hh = 0; hh < 8; ++hh)
          if (hh < gq) acc[hh] = fmaf(qsm[hh * D + 2 * c2 + 1], k1, fmaf(qsm[hh * D + 2 * c2], k0, acc[hh]));
      }
    }
#pragma unroll
    for (int hh = 0; hh < 8; ++hh) sc[i * 8 + hh] = valid ? acc[hh] * sm : -INFINITY;
  }
  __syncthreads();
  // per-head max and sum (thread hh < gq scans the window; the window is small)
  if (tid < gq) {
    float m = -INFINITY;
    for (int i = 0; i < win; ++i) m = fmaxf(m, sc[i * 8 + tid]);
    float l = 0.f;
    for (int i = 0; i < win; ++i) {
      const float s = sc[i * 8 + tid];
      const float p = s == -INFINITY ? 0.f : ex2(s - m);
      sc[i * 8 + tid] = p;
      l += p;
    }
    red[tid] = m;
    red[8 + tid] = l;
  }
  __syncthreads();
  float* part = ws.part;
  const int stride = a.wl.max_splits + 1;
  for (int idx = tid; idx < gq * D; idx += kThreads) {
    const int hh = idx / D, ch = idx % D;
    float acc = 0.f;
    for (int i = 0; i < win; ++i) {
      const float p = sc[i * 8 + hh];
      if (p != 0.f) acc = fmaf(p, __uint_as_float(static_cast<uint32_t>(vwin[(size_t)i * D + ch]) << 16), acc);
    }
    float* pp = part + (((size_t)b * g.Hq + kvh * gq + hh) * stride + 0) * (D + 4);
    pp[4 + ch] = acc;
    if (ch == 0) {
      pp[0] = red[hh];
      pp[1] = red[8 + hh];
    }
  }
}

// ------------------------------------------------------------------ INT2 split
template <int D, int NT, int P>
struct Int2Layout {
  static constexpr int ROW = D / 4;
  static constexpr int SZ = D / 8;
  static constexpr int KSZ = P * ROW;
  static constexpr int VC = KSZ + P * SZ;
  static constexpr int VSZ = VC + P * ROW;
  static constexpr int BLOCK = VSZ + P * SZ;
  static constexpr int PPS = kStageTokens / P;  // pages per stage
  static constexpr int STAGE = PPS * BLOCK;
  static constexpr int GROUPS = D / 32;
  static constexpr int KT = D / 16;             // QK k-tiles
  static constexpr int MT = D / 16;             // PV m-tiles
};

template <int D, int NT, int P>
__global__ void __launch_bounds__(kThreads) decode_splitk_kernel(DecodeArgs a) {
  using Lay = Int2Layout<D, NT, P>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stage_buf = smem;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * Lay::STAGE);
  int* stage_valid = reinterpret_cast<int*>(bars + kStages);

  const Geom& g = a.g;
  const int b = blockIdx.z, kvh = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int gq = g.gq();
  const int n = a.seq_lens[b];
  if (!seq_len_ok(a, n)) {
    if (tid == 0 && blockIdx.x == 0) flag_error(a.status, kDevBadLen);
    pdl_launch_dependents();
    return;
  }
  if (blockIdx.x == 0) {
    const int req = a.req_slot[b];
    if (req < 0 || req >= g.max_req) {
      if (tid == 0) flag_error(a.status, kDevBadSlot);
      pdl_launch_dependents();
      return;
    }
    pdl_wait();
    window_split<D, NT>(a, b, kvh, reinterpret_cast<float*>(smem));
    pdl_launch_dependents();
    return;
  }
  const int split = blockIdx.x - 1;
  const int h_end = n - g.W;
  if (h_end <= g.S) { pdl_launch_dependents(); return; }
  const int n_hist_pages = (h_end - 1) / P + 1;
  const int pg0 = split * a.wl.pages_per_split;
  if (pg0 >= n_hist_pages) { pdl_launch_dependents(); return; }
  const int pg1 = min(pg0 + a.wl.pages_per_split, n_hist_pages);
  const int n_iters = (pg1 - pg0 + Lay::PPS - 1) / Lay::PPS;

  const int* bt = a.block_table + (size_t)b * a.bt_stride;
  const uint8_t* pool_l = a.pool + (size_t)a.layer * g.layer_pool_bytes();

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  __syncthreads();

  auto issue = [&](int it) {
    const int s = it % kStages;
    uint32_t bytes = 0;
    int mask = 0;
    int pages[Lay::PPS];
#pragma unroll
    for (int i = 0; i < Lay::PPS; ++i) {
      const int lp = pg0 + it * Lay::PPS + i;
      pages[i] = -1;
      if (lp < pg1) {
        const int pid = (lp < a.bt_stride && lp < g.max_pages_per_req) ? bt[lp] : -1;
        if (pid >= 0 && pid < g.num_pages) {
          pages[i] = pid;
          bytes += Lay::BLOCK;
          mask |= 1 << i;
        } else {
          flag_error(a.status, kDevBadPage);
        }
      }
    }
    stage_valid[s] = mask;
    mbar_arrive_expect_tx(&bars[s], bytes);
#pragma unroll
    for (int i = 0; i < Lay::PPS; ++i) {
      if (pages[i] >= 0) {
        const uint8_t* src = pool_l + ((size_t)pages[i] * g.Hkv + kvh) * Lay::BLOCK;
        bulk_g2s(stage_buf + s * Lay::STAGE + i * Lay::BLOCK, src, Lay::BLOCK, &bars[s]);
      }
    }
  };

  if (tid == 0) {
    for (int it = 0; it < kStages && it < n_iters; ++it) issue(it);
  }

  // query side (written by q_rotate): wait for the previous grid
  pdl_wait();
  WsView ws = ws_view(a);
  uint32_t qb[NT][Lay::KT][2];
  float qscale[NT];
  float qg[NT][Lay::GROUPS];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const bool col_ok = (nt * 4 + (gid >> 1)) < gq;
#pragma unroll
    for (int kk = 0; kk < Lay::KT; ++kk) {
      const uint2 f = ws.qfrag[((((size_t)b * g.Hkv + kvh) * NT + nt) * Lay::KT + kk) * 32 + lane];
      qb[nt][kk][0] = col_ok ? f.x : 0u;
      qb[nt][kk][1] = col_ok ? f.y : 0u;
    }
    const int hh = nt * 4 + tig;
    const float* aux = ws.qaux + ((size_t)b * g.Hq + kvh * gq + min(hh, gq - 1)) * 8;
    qscale[nt] = hh < gq ? aux[0] : 0.f;
#pragma unroll
    for (int gi = 0; gi < Lay::GROUPS; ++gi) qg[nt][gi] = hh < gq ? aux[1 + gi] : 0.f;
  }

  const float sm_log2 = kLog2e * rsqrtf((float)D);
  float m_run[NT], l_run[NT];
  float acc[NT][Lay::MT][4];
  float zacc[NT][Lay::GROUPS];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt] = -INFINITY;
    l_run[nt] = 0.f;
#pragma unroll
    for (int mt = 0; mt < Lay::MT; ++mt)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[nt][mt][r] = 0.f;
#pragma unroll
    for (int gi = 0; gi < Lay::GROUPS; ++gi) zacc[nt][gi] = 0.f;
  }

  // rows of this lane inside a 16-token block (token order sigma(k) = k/2 + 8*(k%2))
  const int ra = (gid >> 1) + 8 * (gid & 1);      // sigma(gid)
  const int rb = 4 + (gid >> 1) + 8 * (gid & 1);  // sigma(gid + 8)
  const int w_off = 16 * warp;                    // this warp's block inside the stage
  const int pi = w_off / P, slot0 = w_off % P;

  bool aborted = false;
  int it_fail = 0;
  for (int it = 0; it < n_iters; ++it) {
    const int s = it % kStages;
    const bool ok = mbar_wait_bounded(&bars[s], (it / kStages) & 1, a.status);
    if (ok) {
      const int valid_mask = stage_valid[s];
      const bool page_ok = (valid_mask >> pi) & 1;
      const int tb = (pg0 + it * Lay::PPS) * P + w_off;  // absolute token of row 0 of the block
      const uint8_t* buf = stage_buf + s * Lay::STAGE + pi * Lay::BLOCK;
      // ---------------- QK
      uint32_t ua[2 * Lay::GROUPS * 2], ub[2 * Lay::GROUPS * 2];  // D/8 pairs per row
      {
        const uint8_t* kc = buf;
        if constexpr (D == 128) {
          const uint2 wa = *reinterpret_cast<const uint2*>(kc + (slot0 + ra) * Lay::ROW + tig * 8);
          const uint2 wb = *reinterpret_cast<const uint2*>(kc + (slot0 + rb) * Lay::ROW + tig * 8);
          uint32_t t8[8];
          unpack_word(wa.x, t8);
#pragma unroll
          for (int x = 0; x < 8; ++x) ua[x] = t8[x];
          unpack_word(wa.y, t8);
#pragma unroll
          for (int x = 0; x < 8; ++x) ua[8 + x] = t8[x];
          unpack_word(wb.x, t8);
#pragma unroll
          for (int x = 0; x < 8; ++x) ub[x] = t8[x];
          unpack_word(wb.y, t8);
#pragma unroll
          for (int x = 0; x < 8; ++x) ub[8 + x] = t8[x];
        } else {
          const uint32_t wa = *reinterpret_cast<const uint32_t*>(kc + (slot0 + ra) * Lay::ROW + tig * 4);
          const uint32_t wb = *reinterpret_cast<const uint32_t*>(kc + (slot0 + rb) * Lay::ROW + tig * 4);
          uint32_t t8[8];
          unpack_word(wa, t8);
#pragma unroll
          for (int x = 0; x < 8; ++x) ua[x] = t8[x];
          unpack_word(wb, t8);
#pragma unroll
          for (int x = 0; x < 8; ++x) ub[x] = t8[x];
        }
      }
      float sca[NT], scb[NT];
      {
        const uint32_t* kszA = reinterpret_cast<const uint32_t*>(buf + Lay::KSZ + (slot0 + ra) * Lay::SZ);
        const uint32_t* kszB = reinterpret_cast<const uint32_t*>(buf + Lay::KSZ + (slot0 + rb) * Lay::SZ);
        uint32_t sza[Lay::GROUPS], szb[Lay::GROUPS];
#pragma unroll
        for (int gi = 0; gi < Lay::GROUPS; ++gi) {
          sza[gi] = kszA[gi];
          szb[gi] = kszB[gi];
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          float da = 0.f, db = 0.f, za = 0.f, zb = 0.f;
#pragma unroll
          for (int gi = 0; gi < Lay::GROUPS; ++gi) {
            float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kt = 0; kt < 2; ++kt) {
              const int p8 = 4 * gi + 2 * kt;
              mma_f16(c, ua[p8], ub[p8], ua[p8 + 1], ub[p8 + 1], qb[nt][2 * gi + kt][0], qb[nt][2 * gi + kt][1]);
            }
            da = fmaf(bf16_lo(sza[gi]), c[0] + c[1], da);
            db = fmaf(bf16_lo(szb[gi]), c[2] + c[3], db);
            za = fmaf(bf16_hi(sza[gi]), qg[nt][gi], za);
            zb = fmaf(bf16_hi(szb[gi]), qg[nt][gi], zb);
          }
          sca[nt] = fmaf(da, qscale[nt], za) * sm_log2;
          scb[nt] = fmaf(db, qscale[nt], zb) * sm_log2;
        }
      }
      const int ta = tb + ra, tbk = tb + rb;
      const bool va = page_ok && ta >= g.S && ta < h_end;
      const bool vb = page_ok && tbk >= g.S && tbk < h_end;
      // ---------------- online softmax (per head: lanes sharing tig)
      float pa[NT], pb[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        const float s_a = va ? sca[nt] : -INFINITY;
        const float s_b = vb ? scb[nt] : -INFINITY;
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
        for (int mt = 0; mt < Lay::MT; ++mt)
#pragma unroll
          for (int r = 0; r < 4; ++r) acc[nt][mt][r] *= alpha;
#pragma unroll
        for (int gi = 0; gi < Lay::GROUPS; ++gi) zacc[nt][gi] *= alpha;
      }
      // ---------------- zero term of the values (rows ra, rb)
      {
        const uint32_t* vszA = reinterpret_cast<const uint32_t*>(buf + Lay::VSZ + (slot0 + ra) * Lay::SZ);
        const uint32_t* vszB = reinterpret_cast<const uint32_t*>(buf + Lay::VSZ + (slot0 + rb) * Lay::SZ);
#pragma unroll
        for (int gi = 0; gi < Lay::GROUPS; ++gi) {
          const float z_a = bf16_hi(vszA[gi]);
          const float z_b = bf16_hi(vszB[gi]);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            if (pa[nt] > 0.f) zacc[nt][gi] = fmaf(pa[nt], z_a, zacc[nt][gi]);
            if (pb[nt] > 0.f) zacc[nt][gi] = fmaf(pb[nt], z_b, zacc[nt][gi]);
          }
        }
      }
      // ---------------- PV
      {
        // value-side A fragments: rows k in {2tig, 2tig+1, 2tig+8, 2tig+9} are tokens
        // sigma(k) = tig, tig+8, tig+4, tig+12; this lane reads word gid (D=128) of each.
        const uint8_t* vc = buf + Lay::VC;
        uint32_t ux[D / 8], uy[D / 8];
        if constexpr (D == 128) {
          const uint32_t w0 = *reinterpret_cast<const uint32_t*>(vc + (slot0 + tig) * Lay::ROW + gid * 4);
          const uint32_t w1 = *reinterpret_cast<const uint32_t*>(vc + (slot0 + tig + 8) * Lay::ROW + gid * 4);
          const uint32_t w8 = *reinterpret_cast<const uint32_t*>(vc + (slot0 + tig + 4) * Lay::ROW + gid * 4);
          const uint32_t w9 = *reinterpret_cast<const uint32_t*>(vc + (slot0 + tig + 12) * Lay::ROW + gid * 4);
          uint32_t t8[8];
          unpack_word_bf16(prmt(w0, w1, 0x5410), t8);
#pragma unroll
          for (int x = 0; x < 8; ++x) ux[x] = t8[x];
          unpack_word_bf16(prmt(w0, w1, 0x7632), t8);
#pragma unroll
          for (int x = 0; x < 8; ++x) ux[8 + x] = t8[x];
          unpack_word_bf16(prmt(w8, w9, 0x5410), t8);
#pragma unroll
          for (int x = 0; x < 8; ++x) uy[x] = t8[x];
          unpack_word_bf16(prmt(w8, w9, 0x7632), t8);
#pragma unroll
          for (int x = 0; x < 8; ++x) uy[8 + x] = t8[x];
        } else {
          const uint32_t sel = (gid & 1) ? 0x7632u : 0x5410u;
          const int wo = (gid >> 1) * 4;
          const uint32_t w0 = *reinterpret_cast<const uint32_t*>(vc + (slot0 + tig) * Lay::ROW + wo);
          const uint32_t w1 = *reinterpret_cast<const uint32_t*>(vc + (slot0 + tig + 8) * Lay::ROW + wo);
          const uint32_t w8 = *reinterpret_cast<const uint32_t*>(vc + (slot0 + tig + 4) * Lay::ROW + wo);
          const uint32_t w9 = *reinterpret_cast<const uint32_t*>(vc + (slot0 + tig + 12) * Lay::ROW + wo);
          unpack_word_bf16(prmt(w0, w1, sel), ux);
          unpack_word_bf16(prmt(w8, w9, sel), uy);
        }
        const uint32_t* vs0 = reinterpret_cast<const uint32_t*>(buf + Lay::VSZ + (slot0 + tig) * Lay::SZ);
        const uint32_t* vs1 = reinterpret_cast<const uint32_t*>(buf + Lay::VSZ + (slot0 + tig + 8) * Lay::SZ);
        const uint32_t* vs8 = reinterpret_cast<const uint32_t*>(buf + Lay::VSZ + (slot0 + tig + 4) * Lay::SZ);
        const uint32_t* vs9 = reinterpret_cast<const uint32_t*>(buf + Lay::VSZ + (slot0 + tig + 12) * Lay::SZ);
        const int src0 = (2 * tig) * 4 + (gid >> 1);
        const int src1 = (2 * tig + 1) * 4 + (gid >> 1);
        const bool lo_lane = (gid & 1) != 0;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const float p0 = __shfl_sync(0xffffffffu, pa[nt], src0);
          const float p1 = __shfl_sync(0xffffffffu, pa[nt], src1);
          const float p8v = __shfl_sync(0xffffffffu, pb[nt], src0);
          const float p9 = __shfl_sync(0xffffffffu, pb[nt], src1);
#pragma unroll
          for (int gi = 0; gi < Lay::GROUPS; ++gi) {
            float wv[4];
            const float pr[4] = {p0, p1, p8v, p9};
            const uint32_t szr[4] = {vs0[gi], vs1[gi], vs8[gi], vs9[gi]};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float w = pr[u] > 0.f ? pr[u] * bf16_lo(szr[u]) : 0.f;
              const __nv_bfloat16 hi = __float2bfloat16_rn(w);
              const float hif = __bfloat162float(hi);
              wv[u] = lo_lane ? (w - hif) : hif;
            }
            const uint32_t b0 = pack_bf162(wv[0], wv[1]);
            const uint32_t b1 = pack_bf162(wv[2], wv[3]);
#pragma unroll
            for (int mq = 0; mq < 2; ++mq) {
              const int mt = 2 * gi + mq;
              mma_bf16(acc[nt][mt], ux[2 * mt], ux[2 * mt + 1], uy[2 * mt], uy[2 * mt + 1], b0, b1);
            }
          }
        }
      }
    }
    // every warp is done with stage s (uniform abort decision)
    aborted = __syncthreads_or(!ok) != 0;
    if (aborted) {
      it_fail = it;
      break;
    }
    if (tid == 0 && it + kStages < n_iters) issue(it + kStages);
  }
  if (aborted) {
    // drain copies still in flight before the CTA exits, again bounded
    if (tid == 0) {
      const int last = min(n_iters, it_fail + kStages);
      for (int it = it_fail; it < last; ++it) (void)mbar_wait_bounded(&bars[it % kStages], (it / kStages) & 1, nullptr);
    }
    __syncthreads();
    pdl_launch_dependents();
    return;
  }
  pdl_launch_dependents();

  // ---------------- per-warp finalisation
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    l_run[nt] += __shfl_xor_sync(0xffffffffu, l_run[nt], 4);
    l_run[nt] += __shfl_xor_sync(0xffffffffu, l_run[nt], 8);
    l_run[nt] += __shfl_xor_sync(0xffffffffu, l_run[nt], 16);
#pragma unroll
    for (int gi = 0; gi < Lay::GROUPS; ++gi) {
      zacc[nt][gi] += __shfl_xor_sync(0xffffffffu, zacc[nt][gi], 4);
      zacc[nt][gi] += __shfl_xor_sync(0xffffffffu, zacc[nt][gi], 8);
      zacc[nt][gi] += __shfl_xor_sync(0xffffffffu, zacc[nt][gi], 16);
    }
  }
  // cross-warp merge through shared memory (the stage ring is free now)
  float* wm = reinterpret_cast<float*>(smem);   // [4][8]
  float* wl = wm + 32;                          // [4][8]
  float* wacc = wl + 32;                        // [4][8][D]
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int hh = nt * 4 + tig;
    if (hh < gq) {
      if (gid == 0) {
        wm[warp * 8 + hh] = m_run[nt];
        wl[warp * 8 + hh] = l_run[nt];
      }
#pragma unroll
      for (int mt = 0; mt < Lay::MT; ++mt) {
        const int ch_a = 16 * mt + gid, ch_b = ch_a + 8;
        // channel ch of the V row sits in slot s = (ch mod 64) / 8 with bit position vpos(s)
        const int sa = (ch_a & 63) >> 3, sb = (ch_b & 63) >> 3;
        const float va = ldexpf(acc[nt][mt][0] + acc[nt][mt][1], 7 - slot_pos_bf16(sa)) + zacc[nt][ch_a / 32];
        const float vb = ldexpf(acc[nt][mt][2] + acc[nt][mt][3], 7 - slot_pos_bf16(sb)) + zacc[nt][ch_b / 32];
        wacc[(warp * 8 + hh) * D + ch_a] = va;
        wacc[(warp * 8 + hh) * D + ch_b] = vb;
      }
    }
  }
  __syncthreads();
  const int stride = a.wl.max_splits + 1;
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
    float* pp = ws.part + (((size_t)b * g.Hq + kvh * gq + hh) * stride + blockIdx.x) * (D + 4);
    pp[4 + ch] = accv;
    if (ch == 0) {
      pp[0] = M;
      pp[1] = L;
    }
  }
}

// ------------------------------------------------------------------ combine
// grid (Hq, B), block 128.  Merges the window partial (plain basis) and the
// INT2 partials (rotated basis), applies R_V^T once, divides by l.
template <int D>
__global__ void __launch_bounds__(kThreads) decode_combine_kernel(DecodeArgs a) {
  pdl_wait();
  const Geom& g = a.g;
  const int h = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  __shared__ float rot[D];
  __shared__ float rotated_out[D];
  __shared__ float wts[kMaxSplits + 1];
  __shared__ float s_l;
  WsView ws = ws_view(a);
  const int n = a.seq_lens[b];
  const int nsp = seq_len_ok(a, n) ? min(splits_for(a, n), kMaxSplits) : 0;
  const int stride = a.wl.max_splits + 1;
  const float* base = ws.part + ((size_t)b * g.Hq + h) * stride * (D + 4);
  if (warp == 0) {
    float M = -INFINITY;
    for (int i = lane; i <= nsp; i += 32) M = fmaxf(M, base[(size_t)i * (D + 4)]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float L = 0.f;
    for (int i = lane; i <= nsp; i += 32) {
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
  float plain = 0.f;
  if (tid < D) {
    float r = 0.f;
    for (int i = 1; i <= nsp; ++i) r = fmaf(wts[i], base[(size_t)i * (D + 4) + 4 + tid], r);
    rot[tid] = r;
    plain = wts[0] * base[4 + tid];
  }
  __syncthreads();
  // (rot R_V^T)_j = sum_k rot_k R_V[j][k]; warp w handles rows j = w, w + 4, ...
  for (int j = warp; j < D; j += kThreads / 32) {
    float s = 0.f;
    for (int k = lane; k < D; k += 32) s = fmaf(rot[k], a.R_V[(size_t)j * D + k], s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) rotated_out[j] = s;
  }
  __syncthreads();
  if (tid < D) {
    const float inv = s_l > 0.f ? 1.f / s_l : 0.f;
    const float o = (plain + rotated_out[tid]) * inv;
    const size_t oi = ((size_t)b * g.Hq + h) * D + tid;
    if (a.out_dtype == kDtypeBF16) {
      __nv_bfloat16 hb = __float2bfloat16_rn(o);
      static_cast<uint16_t*>(a.out)[oi] = *reinterpret_cast<uint16_t*>(&hb);
    } else {
      static_cast<float*>(a.out)[oi] = o;
    }
  }
}

template <int D, int NT, int P>
int launch_splitk_t(const DecodeArgs& a, cudaStream_t s, bool pdl) {
  using Lay = Int2Layout<D, NT, P>;
  size_t smem = kStages * Lay::STAGE + kStages * 8 + kStages * 4;
  const size_t win_smem = (8 * D + a.g.window() * 8 + 64) * sizeof(float);
  const size_t merge_smem = (64 + 4 * 8 * D) * sizeof(float);
  if (win_smem > smem) smem = win_smem;
  if (merge_smem > smem) smem = merge_smem;
  smem = (smem + 127) & ~size_t(127);
  auto kern = decode_splitk_kernel<D, NT, P>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.wl.max_splits + 1, a.g.Hkv, a.batch);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  e = cudaLaunchKernelEx(&cfg, kern, a);
  return (int)e;
}

template <int D, int NT>
int launch_splitk_p(const DecodeArgs& a, cudaStream_t s, bool pdl) {
  switch (a.g.P) {
    case 16: return launch_splitk_t<D, NT, 16>(a, s, pdl);
    case 32: return launch_splitk_t<D, NT, 32>(a, s, pdl);
    default: return launch_splitk_t<D, NT, 64>(a, s, pdl);
  }
}

}  // namespace

int static_decode_scratch(void** out, size_t* capacity) {
  constexpr int kMaxDevices = 64;
  static std::mutex mu;
  static void* ptrs[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  if (dev < 0 || dev >= kMaxDevices) return (int)cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);  // with this device current
    if (e != cudaSuccess) return (int)e;
    ptrs[dev] = p;
  }
  *out = ptrs[dev];
  *capacity = kStaticScratchBytes;
  return 0;
}

int launch_q_rotate(const DecodeArgs& a, void* stream) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  dim3 grid(a.g.Hq, a.batch);
  if (a.g.D == 128) q_rotate_kernel<128><<<grid, kThreads, 0, s>>>(a);
  else q_rotate_kernel<64><<<grid, kThreads, 0, s>>>(a);
  return (int)cudaGetLastError();
}

int launch_decode_splitk(const DecodeArgs& a, void* stream, bool pdl) {
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int nt = a.wl.nt;
  if (a.g.D == 128) return nt == 2 ? launch_splitk_p<128, 2>(a, s, pdl) : launch_splitk_p<128, 1>(a, s, pdl);
  return nt == 2 ? launch_splitk_p<64, 2>(a, s, pdl) : launch_splitk_p<64, 1>(a, s, pdl);
}

int launch_decode_combine(const DecodeArgs& a, void* stream, bool pdl) {
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
  if (a.g.D == 128) return (int)cudaLaunchKernelEx(&cfg, decode_combine_kernel<128>, a);
  return (int)cudaLaunchKernelEx(&cfg, decode_combine_kernel<64>, a);
}

}  // namespace oscar
