// Device helpers shared by the OSCAR kernels (sm_103a).
//
// Everything here is hand-written inline PTX or plain CUDA: mbarrier phase
// waits (always bounded by %globaltimer so a lost copy can never hang the GPU),
// non-multicast bulk global->shared copies, warp-level f16 MMA, and the
// magic-number unpack of 2-bit codes into f16 pairs.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "oscar_internal.h"

namespace oscar {

// Raise a kernel's dynamic shared-memory limit once per (kernel, device) (the
// first launch on a device), so that later launches, including ones recorded
// into a CUDA graph, issue nothing but the launch itself.  max_carveout: also ask
// for the largest shared-memory share of the SM's L1/shared storage, for kernels
// whose resident CTAs per SM need it (the CUDA runtime's default carveout may leave room
// for fewer).
inline cudaError_t ensure_smem_limit_ptr(const void* kern, size_t bytes, bool max_carveout = false) {
  struct Entry { const void* k; int dev; size_t bytes; };
  static std::mutex mu;
  static Entry table[256];
  static int used = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  for (int i = 0; i < used; ++i)
    if (table[i].k == kern && table[i].dev == dev && table[i].bytes >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  if (max_carveout) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
  }
  for (int i = 0; i < used; ++i)
    if (table[i].k == kern && table[i].dev == dev) { table[i].bytes = bytes; return cudaSuccess; }
  if (used < 256) table[used++] = Entry{kern, dev, bytes};
  return cudaSuccess;
}

template <typename Kernel>
inline cudaError_t ensure_smem_limit(Kernel kern, size_t bytes, bool max_carveout = false) {
  return ensure_smem_limit_ptr(reinterpret_cast<const void*>(kern), bytes, max_carveout);
}

// Launch kern<<<grid, block, smem, s>>>(args...) as a programmatic dependent of the
// kernel before it on the stream when pdl is set (the kernel waits with pdl_wait()
// before it touches what that kernel writes).
template <typename Kernel, typename... Args>
inline int launch_pdl(Kernel kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl, const Args&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return (int)cudaLaunchKernelEx(&cfg, kern, args...);
}

__device__ __forceinline__ void flag_error(int* status, int bits) {
  if (status) atomicOr(status, bits);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Ends an mbarrier's life so that its shared memory can hold other data.
__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase with the given parity to complete, giving up after
// kWaitLimitNs.  On give-up the status word gets OSCAR_DEV_TIMEOUT and false
// is returned; callers then stop issuing work and drain.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      flag_error(status, kDevTimeout);
      return false;
    }
  }
}

// try_wait with a suspend-time hint: a thread whose phase has not completed is
// suspended (it issues nothing) until the phase completes or about hint_ns pass.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// mbar_wait_bounded for warps that wait while others work: the waiting thread
// sleeps in the barrier (no spinning that would take issue slots from the warps
// it waits for) and reads the timer only every 16 retries.  Same limit and
// timeout behaviour as mbar_wait_bounded.
__device__ __forceinline__ bool mbar_wait_sleep_bounded(uint64_t* bar, uint32_t parity, int* status) {
  if (mbar_try_wait_sleep(bar, parity, 1000u)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t k = 1;; ++k) {
    if (mbar_try_wait_sleep(bar, parity, 1000u)) return true;
    if ((k & 15) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) {
      flag_error(status, kDevTimeout);
      return false;
    }
  }
}

// Non-multicast bulk copy global -> this CTA's shared memory, completion
// signalled on an mbarrier (complete_tx).  Both addresses 16-byte aligned,
// bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// L2 policy for data read once per step (the INT2 page stream): evict first, so
// that streaming the cache does not push small reused data (rotations, window
// slabs, workspaces) out of L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// bulk_g2s with an L2 cache-eviction policy from l2_evict_first_policy().
__device__ __forceinline__ void bulk_g2s_hint(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Bring bytes of global memory into L2 ahead of a later read (no data reaches the
// SM; L2 is the point of coherence, so a write that lands later is what that read
// sees).  Address 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* gsrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(gsrc), "r"(bytes) : "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before its
// later async-proxy ones (a bulk copy into a buffer the warp has just read).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ PDL
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------ MMA
// D = A(16x16, row) * B(16x8, col) + D, f16 inputs, f32 accumulate.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------ code unpack
// A 32-bit word holds 8 slot pairs: slot x has one code at bits 2x and one at
// bits 16+2x.  Slots 0..4 are read in place (positions 0,2,4,6,8), slots 5..7
// after a right shift by 6 (positions 4,6,8).  OR-ing a code c sitting at
// mantissa bits [pos, pos+2) into the f16 pattern of 1.0 gives 1 + c*2^(pos-10)
// exactly; subtracting 1.0 leaves c * 2^(pos-10), also exact.  The 2^(10-pos)
// factor is folded into the other MMA operand (query side) or into the final
// per-channel scaling (value side).
__host__ __device__ constexpr int slot_pos(int x) { return x < 5 ? 2 * x : 2 * x - 6; }

__device__ __forceinline__ uint32_t hsub2_one(uint32_t v) {
  const __half2 x = *reinterpret_cast<const __half2*>(&v);
  const __half2 r = __hsub2(x, __half2half2(__ushort_as_half(0x3C00)));
  return *reinterpret_cast<const uint32_t*>(&r);
}

template <int X>
__device__ __forceinline__ uint32_t unpack_slot(uint32_t w, uint32_t w6) {
  constexpr int pos = slot_pos(X);
  constexpr uint32_t mask = (3u << pos) | (3u << (16 + pos));
  const uint32_t src = X < 5 ? w : w6;
  return hsub2_one((src & mask) | 0x3C003C00u);
}

__device__ __forceinline__ void unpack_word(uint32_t w, uint32_t (&o)[8]) {
  const uint32_t w6 = w >> 6;
  o[0] = unpack_slot<0>(w, w6);
  o[1] = unpack_slot<1>(w, w6);
  o[2] = unpack_slot<2>(w, w6);
  o[3] = unpack_slot<3>(w, w6);
  o[4] = unpack_slot<4>(w, w6);
  o[5] = unpack_slot<5>(w, w6);
  o[6] = unpack_slot<6>(w, w6);
  o[7] = unpack_slot<7>(w, w6);
}

// BF16 variant: bfloat16 keeps 7 stored mantissa bits, so codes are read at
// positions 0, 2, 4 only: slots 0..2 in place, 3..5 after >> 6, 6..7 after
// >> 12.  (1.0 | c << pos) - 1.0 = c * 2^(pos-7), exact in bfloat16.
__host__ __device__ constexpr int slot_pos_bf16(int x) { return x < 3 ? 2 * x : (x < 6 ? 2 * (x - 3) : 2 * (x - 6)); }

__device__ __forceinline__ uint32_t bsub2_one(uint32_t v) {
  const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&v);
  const __nv_bfloat162 r = __hsub2(x, __bfloat162bfloat162(__ushort_as_bfloat16(0x3F80)));
  return *reinterpret_cast<const uint32_t*>(&r);
}

template <int X>
__device__ __forceinline__ uint32_t unpack_slot_bf16(uint32_t w, uint32_t w6, uint32_t w12) {
  constexpr int pos = slot_pos_bf16(X);
  constexpr uint32_t mask = (3u << pos) | (3u << (16 + pos));
  const uint32_t src = X < 3 ? w : (X < 6 ? w6 : w12);
  return bsub2_one((src & mask) | 0x3F803F80u);
}

__device__ __forceinline__ void unpack_word_bf16(uint32_t w, uint32_t (&o)[8]) {
  const uint32_t w6 = w >> 6, w12 = w >> 12;
  o[0] = unpack_slot_bf16<0>(w, w6, w12);
  o[1] = unpack_slot_bf16<1>(w, w6, w12);
  o[2] = unpack_slot_bf16<2>(w, w6, w12);
  o[3] = unpack_slot_bf16<3>(w, w6, w12);
  o[4] = unpack_slot_bf16<4>(w, w6, w12);
  o[5] = unpack_slot_bf16<5>(w, w6, w12);
  o[6] = unpack_slot_bf16<6>(w, w6, w12);
  o[7] = unpack_slot_bf16<7>(w, w6, w12);
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) { return __byte_perm(a, b, sel); }

// ------------------------------------------------------------------ scaled code operands
// f16 pair of slot X of a code word (w6 = w >> 6): -(1 + c * 2^(pos-10)) in each
// half, the f16 pattern of -1.0 with the code OR-ed into its mantissa.
// magic is kCodeMagic, passed in from the host so that it stays in a register
// and (w & mask) | magic is a single LOP3 with the mask as its immediate.
template <int X>
__device__ __forceinline__ uint32_t magic_slot(uint32_t w, uint32_t w6, uint32_t magic) {
  constexpr int pos = slot_pos(X);
  constexpr uint32_t mask = (3u << pos) | (3u << (16 + pos));
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(X < 5 ? w : w6), "n"(mask), "r"(magic));  // (a & b) | c
  return r;
}

// x * N + N = S * c * 2^(pos-10) for x = -(1 + c * 2^(pos-10)) and N = -S: one
// fused f16 multiply-add per pair, with no separate negation.  The result is
// exact whenever it is an f16 normal number: S carries at most 8 significant
// bits (a BF16 value times a power of two) and c * 2^(pos-10) at most 2.
__device__ __forceinline__ uint32_t scale_codes(uint32_t x, uint32_t n2) {
  const __half2 xv = *reinterpret_cast<const __half2*>(&x);
  const __half2 nv = *reinterpret_cast<const __half2*>(&n2);
  const __half2 r = __hfma2(xv, nv, nv);
  return *reinterpret_cast<const uint32_t*>(&r);
}

// A (scale, zero) word holds the BF16 scale in its low half and the BF16 zero
// in its high half.  neg_scale_times_pow2 returns -scale * 2^k and
// zero_times_pow2 zero * 2^k as float32, by adding k to the exponent field
// (k23 = k << 23, k >= 0; the scale is never negative, so adding the sign bit
// negates it).  A zero field turns into +-2^(k-127), below every f16 number,
// which converts to 0.
__device__ __forceinline__ float neg_scale_times_pow2(uint32_t w, uint32_t k23) {
  return __uint_as_float(w * 65536u + (k23 + 0x80000000u));
}
__device__ __forceinline__ float zero_times_pow2(uint32_t w, uint32_t k23) {
  return __uint_as_float((w & 0xFFFF0000u) + k23);
}
// scale * 2^k as float32 (k23 = k << 23, k >= 0).
__device__ __forceinline__ float scale_times_pow2(uint32_t w, uint32_t k23) {
  return __uint_as_float(w * 65536u + k23);
}

// The codes of slot X of a packed word as an f16 pair of subnormals c * 2^(pos - 24):
// exact tensor-core operands with no offset term, so a product with q * 2^(e + 10 - pos)
// is exactly c * q * 2^(e - 14) and the group's scale can be applied after the MMA.
template <int X>
__device__ __forceinline__ uint32_t subnormal_slot(uint32_t w, uint32_t w6) {
  constexpr int pos = slot_pos(X);
  constexpr uint32_t mask = (3u << pos) | (3u << (16 + pos));
  return (X < 5 ? w : w6) & mask;
}

__device__ __forceinline__ uint32_t pack_half2(float lo_elem, float hi_elem) {
  __half2 h = __floats2half2_rn(lo_elem, hi_elem);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint32_t pack_bf162(float lo_elem, float hi_elem) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo_elem, hi_elem);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// 2^x with the hardware approximation (ex2.approx.ftz: relative error ~2^-22,
// ex2(-inf) = 0); used for softmax weights, which tolerate it.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float warp_max_xor(float v, int lane_mask) {
  return fmaxf(v, __shfl_xor_sync(0xffffffffu, v, lane_mask));
}

}  // namespace oscar
