// Decode workspace view and the query rotation of one CTA, shared by the
// decode kernels (kernels_decode.cu) and the fused step's preparation kernel
// (kernels_write.cu).  Included inside namespace oscar's anonymous namespace.
#pragma once

// ------------------------------------------------------------------ workspace views
struct WsView {
  uint2* qfrag;   // [B][Hkv][NT][D/16][32]
  float* qaux;    // [B][Hq][8]: [0] = 2^-e_h, [1 + g] = Q_g
  float* qplain;  // [B][Hq][D]
  float* part;    // [B][Hq][win_chunks + max_splits][D + 4]: [0] m (log2 domain), [1] l, [4..] acc
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

// Destinations of one (request, kv head)'s query side: the query-side MMA fragments
// [NT][D/16][32 lanes], per head 2^-e_h and the group sums Q_g [gq][8], and q as
// float32 [gq][D] (may be null).  In the decode workspace (q_rotate kernel, step
// prep) or in the shared memory of a CTA that rotates its own query.
struct QOut {
  uint2* qfrag;
  float* qaux;
  float* qplain;
};

__device__ __forceinline__ QOut q_out_ws(const DecodeArgs& a, int kvh, int b) {
  WsView ws = ws_view(a);
  const int gq = a.g.gq();
  QOut o;
  o.qfrag = ws.qfrag + (((size_t)b * a.g.Hkv + kvh) * a.wl.nt) * (a.g.D / 16) * 32;
  o.qaux = ws.qaux + ((size_t)b * a.g.Hq + (size_t)kvh * gq) * 8;
  o.qplain = ws.qplain + ((size_t)b * a.g.Hq + (size_t)kvh * gq) * a.g.D;
  return o;
}

// ------------------------------------------------------------------ query-side fragments
// Power-of-two exponent e of a head: |q'|_inf <= ||q||_2 = nrm (R_K is orthogonal), and
// |q'| * 2^e < 32, so that q' * 2^e * 2^(10 - pos) <= 1024 x 32 stays below the f16 maximum.
__device__ __forceinline__ int q_head_exp(float nrm) {
  int e = 0;
  if (nrm > 0.f) {
    int E;
    frexpf(nrm, &E);  // nrm * (1 + rounding) < 2^E
    e = 5 - E;
  }
  return e;
}

// One entry of the query-side MMA fragments: head hh of the kv head's gq, channel
// group grp (k-tiles 2 grp, 2 grp + 1), sub in [0, 16) = (k-tile, hi|lo half, tig).
// qg: q'_hh over the group's 32 channels; e: the head's exponent.  Writes the
// register pair of lane ln in k-tile kk of plane `plane` of qfrag [NT][D/16][32].
template <int D>
__device__ __forceinline__ void q_frag_entry(const float* qg, int hh, int grp, int sub, int e, int gq, uint2* qfrag) {
  const int kt = sub >> 3, hl = (sub >> 2) & 1, tig = sub & 3;
  const bool g8 = gq == 8;
  const int gid = g8 ? hh : 2 * (hh & 3) + hl;
  const int plane = g8 ? hl : 0;
  const int ln = gid * 4 + tig;
  const int kk = 2 * grp + kt;
  const int p8 = 4 * grp + 2 * kt;
  uint32_t regs[2];
#pragma unroll
  for (int hpair = 0; hpair < 2; ++hpair) {
    const int ch = 16 * kt + 8 * hpair + 2 * tig;  // channel within the group
    const int pos = slot_pos((p8 + hpair) & 7);
    float v[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const float x = ldexpf(qg[ch + u], e + 10 - pos);
      const __half hi = __float2half_rn(x);
      const float lo = x - __half2float(hi);
      v[u] = hl ? lo : __half2float(hi);
    }
    regs[hpair] = pack_half2(v[0], v[1]);
  }
  qfrag[((size_t)plane * (D / 16) + kk) * 32 + ln] = make_uint2(regs[0], regs[1]);
}

// ------------------------------------------------------------------ q rotate
// One CTA of 128 threads, (kv head kvh, channel group grp, request b): the 32
// rotated channels of group grp, q'_j = sum_i q_i R_K[i][j] for j in
// [32 grp, 32 grp + 32), for every query head of kv head kvh; it writes the
// group sum Q_g and the query-side MMA fragments of its two k-tiles.  The
// power-of-two scale of head h is set from ||q_h||_2, which bounds |q'_h|_inf
// (R_K is orthogonal), so the CTAs of a head need not agree on a maximum.
//
// The loads of the R_K slice (a per-layer constant) are issued before the wait
// on the preceding grid (q may come from it); the CTA lets its own dependents
// launch right after that wait.  sm: shared memory of kQRotSmemFloats<D>() floats.
template <int D>
__host__ __device__ constexpr int kQRotSmemFloats() { return D * 33 + 8 * D + 8 * 32 + 8; }

// pdl: the CTA waits on the preceding grid (after issuing its R_K loads) and lets its
// dependents launch; false when the caller has already waited.
template <int D>
__device__ __forceinline__ void q_rotate_cta(const DecodeArgs& a, int grp, int kvh, int b, float* sm, QOut out,
                                             bool pdl = true) {
  constexpr int T = 128;
  float (*Rs)[33] = reinterpret_cast<float (*)[33]>(sm);          // [D][33]: R_K[:, 32 grp + c], padded
  float (*qs)[D] = reinterpret_cast<float (*)[D]>(sm + D * 33);   // [8][D]
  float (*qr)[32] = reinterpret_cast<float (*)[32]>(sm + D * 33 + 8 * D);
  float* nrm = sm + D * 33 + 8 * D + 8 * 32;
  const Geom& g = a.g;
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int gq = g.gq();
  // R_K column slice: D rows x 32 floats (8 float4 per row), 16-byte loads, all in flight
  {
    const float4* Rg = reinterpret_cast<const float4*>(a.R_K + (size_t)kvh * g.rot_stride());  // this kv head's R_K
    float4 v[D * 8 / T];
#pragma unroll
    for (int u = 0; u < D * 8 / T; ++u) {
      const int idx = t + u * T;  // row idx / 8, float4 idx % 8
      v[u] = __ldg(Rg + (size_t)(idx >> 3) * (D / 4) + grp * 8 + (idx & 7));
    }
#pragma unroll
    for (int u = 0; u < D * 8 / T; ++u) {
      const int idx = t + u * T;
      float* dst = &Rs[idx >> 3][(idx & 7) * 4];
      dst[0] = v[u].x; dst[1] = v[u].y; dst[2] = v[u].z; dst[3] = v[u].w;
    }
    if (pdl) {
      pdl_wait();
      pdl_launch_dependents();
    }
  }
  const size_t qbase = ((size_t)b * g.Hq + (size_t)kvh * gq) * D;
  {
    constexpr int QMAX = 8 * D / T;   // gq <= 8: every load of q in flight at once
    float qv[QMAX];
#pragma unroll
    for (int u = 0; u < QMAX; ++u) {
      const int i = t + u * T;
      qv[u] = i < gq * D ? load_q(a, qbase + i) : 0.f;
    }
#pragma unroll
    for (int u = 0; u < QMAX; ++u) {
      const int i = t + u * T;
      if (i < gq * D) {
        qs[i / D][i % D] = qv[u];
        if (grp == 0 && out.qplain) out.qplain[i] = qv[u];
      }
    }
  }
  __syncthreads();
  // squared norms: warp w sums heads w, w + 4
  for (int hh = warp; hh < gq; hh += T / 32) {
    float ss = 0.f;
    for (int i = lane; i < D; i += 32) ss = fmaf(qs[hh][i], qs[hh][i], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) nrm[hh] = sqrtf(ss);
  }
  // rotation: lane = channel 32 grp + lane, warp w handles heads w, w + 4; four
  // partial sums (inputs i = 4m + r) shorten the dependent chain fourfold
  for (int hh = warp; hh < gq; hh += T / 32) {
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll 8
    for (int i = 0; i < D; i += 4) {
      a0 = fmaf(qs[hh][i], Rs[i][lane], a0);
      a1 = fmaf(qs[hh][i + 1], Rs[i + 1][lane], a1);
      a2 = fmaf(qs[hh][i + 2], Rs[i + 2][lane], a2);
      a3 = fmaf(qs[hh][i + 3], Rs[i + 3][lane], a3);
    }
    const float acc = (a0 + a1) + (a2 + a3);
    qr[hh][lane] = acc;
    float gs = acc;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) gs += __shfl_xor_sync(0xffffffffu, gs, o);
    if (lane == 0) out.qaux[hh * 8 + 1 + grp] = gs;
  }
  __syncthreads();
  // fragments of the two k-tiles of this group: 8 lanes x 2 k-tiles per head
  for (int idx = t; idx < gq * 16; idx += T) {
    const int hh = idx >> 4, sub = idx & 15;
    const int e = q_head_exp(nrm[hh]);
    if (grp == 0 && sub == 0) out.qaux[hh * 8] = ldexpf(1.f, -e);
    q_frag_entry<D>(qr[hh], hh, grp, sub, e, gq, out.qfrag);
  }
}
