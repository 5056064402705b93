// sp_device.cuh — device-side building blocks of the fused reduce + add + RMSNorm + quant
// kernels for sm_103a: 128-bit streaming loads/stores, bf16 unpacking, hardware conversions to
// bf16x2 / e4m3x2 / e2m1x2, mbarrier and bulk-copy primitives, the per-row block reduction and
// the per-row epilogue (new residual, RMSNorm, quantisation, stores).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace spk {

enum { kModeNone = 0, kModeFp8Static = 1, kModeFp8PerToken = 2, kModeNvfp4 = 3 };

// A wait on a shared-memory barrier gives up after this long (ns of %globaltimer); between
// checks a waiting thread sleeps inside mbarrier.try_wait for at most kWaitSleepHintNs.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kWaitSleepHintNs = 100000u;

// Set (atomicOr) by a kernel whose bounded wait ran out; read by sp_device_error().
__device__ unsigned int g_error_flags = 0;
constexpr unsigned int kErrWaitTimeout = 1u;

struct Params {
  const uint16_t* partials;   // bf16 [tp][T_pad][H]
  const uint16_t* residual;   // bf16 [T_pad][H] or null
  const uint16_t* addend;     // bf16 [T_pad][H] or null: added after the reduction
  float partial_scale;        // multiplies the sum of the partials (1 = none)
  int scale_swizzled;         // NVFP4 block scales in the 128x4-tile layout (else row-major)
  int sf_cols;                // swizzled layout: block columns padded to a multiple of 4
  int64_t rows_total;         // rows the CTAs walk: T_pad, or the 128-padded scale rows if more
  const uint16_t* weight;     // bf16 [H]
  const uint16_t* bias;       // bf16 [H] or null
  const float* scale;         // fp32 [1] or null
  void* out;
  void* out_scales;
  uint16_t* residual_out;     // bf16 [T_pad][H]
  int64_t T_pad;
  int64_t T_valid;
  int64_t plane;              // T_pad * H: elements from one partial to the next
  int H;
  int nvec;                   // H / 8: 16-byte vectors in a row
  int tp;
  int nthreads;               // consumer threads per CTA (a multiple of 32, <= 1024)
  float eps;
  int stages;                 // staged kernel: ring depth
  int seg_stride;             // staged kernel: bytes between ring stages (2H rounded up to 128)
  int wb_offset;              // staged kernel: byte offset of the weight/bias copy [2][H] bf16
  int ring_offset;            // staged kernel: byte offset of the ring in dynamic shared memory
  unsigned int* row_counter;  // dynamic schedule: [next claim, CTAs done], zero between calls
  unsigned int* error_word;   // where a timed-out wait is reported: the call's status word, or
                              // else g_error_flags (the device error word)
  uint64_t wait_limit_ns;     // every bounded wait gives up after this long
  int64_t withhold;           // self-test only: CTA 0 skips its ring fill of this issue number
  int split_chunk;            // split rows: 16-byte vectors of a row per CTA of the cluster
  unsigned long long* slot_done;  // dynamic schedule on a slot of the library's counter table:
  unsigned long long slot_seq;    // where and what the launch writes once it has reset the slot
};


// Per-warp slot of the row reduction: sum of squares, max |h*w| and an abort vote.
struct __align__(16) RedSlot {
  float ss;
  float mx;
  int abort;
  int pad;
};

// ---------------------------------------------------------------- global memory
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ uint4 ldg_keep(const void* p) {
  uint4 v;
  asm("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}

__device__ __forceinline__ void stg_stream(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

__device__ __forceinline__ void stg_stream(void* p, uint2 v) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

__device__ __forceinline__ void stg_stream(void* p, uint32_t v) {
  asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// ---------------------------------------------------------------- paired fp32 arithmetic
// Blackwell's packed fp32x2 instructions: each lane is an ordinary IEEE binary32 operation with
// round-to-nearest-even, so (a0, a1) op (b0, b1) equals the two scalar operations bit for bit,
// at half the instruction count.
__device__ __forceinline__ void add2(float& a0, float& a1, float b0, float b1) {
  asm("{\n\t.reg .b64 a, b;\n\t"
      "mov.b64 a, {%0, %1};\n\t"
      "mov.b64 b, {%2, %3};\n\t"
      "add.rn.f32x2 a, a, b;\n\t"
      "mov.b64 {%0, %1}, a;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}

__device__ __forceinline__ void mul2(float& a0, float& a1, float b0, float b1) {
  asm("{\n\t.reg .b64 a, b;\n\t"
      "mov.b64 a, {%0, %1};\n\t"
      "mov.b64 b, {%2, %3};\n\t"
      "mul.rn.f32x2 a, a, b;\n\t"
      "mov.b64 {%0, %1}, a;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}

// (c0, c1) += (a0, a1) * (b0, b1), each lane one fused multiply-add
__device__ __forceinline__ void fma2(float& c0, float& c1, float a0, float a1, float b0,
                                     float b1) {
  asm("{\n\t.reg .b64 a, b, c;\n\t"
      "mov.b64 a, {%2, %3};\n\t"
      "mov.b64 b, {%4, %5};\n\t"
      "mov.b64 c, {%0, %1};\n\t"
      "fma.rn.f32x2 c, a, b, c;\n\t"
      "mov.b64 {%0, %1}, c;\n\t}"
      : "+f"(c0), "+f"(c1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Eight values times one factor.
__device__ __forceinline__ void scale8(float (&v)[8], float f) {
#pragma unroll
  for (int e = 0; e < 8; e += 2) mul2(v[e], v[e + 1], f, f);
}

// ---------------------------------------------------------------- conversions
// bf16 -> fp32 is exact: the bf16 pattern is the top half of the binary32 pattern.
__device__ __forceinline__ void add_bf16x2(uint32_t v, float& a0, float& a1) {
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %2;\n\t"
      "add.rn.f32.bf16 %0, lo, %0;\n\t"
      "add.rn.f32.bf16 %1, hi, %1;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "r"(v));
}
__device__ __forceinline__ void add_bf16x8(const uint4 v, float (&acc)[8]) {
  add_bf16x2(v.x, acc[0], acc[1]);
  add_bf16x2(v.y, acc[2], acc[3]);
  add_bf16x2(v.z, acc[4], acc[5]);
  add_bf16x2(v.w, acc[6], acc[7]);
}

__device__ __forceinline__ void unpack_bf16x8(const uint4 v, float (&f)[8]) {
  f[0] = __uint_as_float(v.x << 16);
  f[1] = __uint_as_float(v.x & 0xFFFF0000u);
  f[2] = __uint_as_float(v.y << 16);
  f[3] = __uint_as_float(v.y & 0xFFFF0000u);
  f[4] = __uint_as_float(v.z << 16);
  f[5] = __uint_as_float(v.z & 0xFFFF0000u);
  f[6] = __uint_as_float(v.w << 16);
  f[7] = __uint_as_float(v.w & 0xFFFF0000u);
}

// Round-to-nearest-even to bf16; `lo` lands in the low 16 bits.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&f)[8]) {
  return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                    pack_bf16x2(f[6], f[7]));
}

// Four values to E4M3 (round to nearest even, saturating to +-448); value i in byte i.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  uint32_t r;
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(r)
      : "f"(a), "f"(b), "f"(c), "f"(d));
  return r;
}

// Eight values to E2M1 (round to nearest even, saturating to +-6); value 2i in the low nibble
// and value 2i+1 in the high nibble of byte i.
__device__ __forceinline__ uint32_t pack_e2m1x8(const float (&v)[8]) {
  uint32_t r;
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
      "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
      : "=r"(r)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return r;
}

// One value to its E4M3 code (low byte).
__device__ __forceinline__ uint32_t e4m3_code(float x) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(x));
  return r & 0xFFu;
}

// Exact value of an E4M3 code (every E4M3 value is an fp16 value).
__device__ __forceinline__ float e4m3_value(uint32_t code) {
  const uint16_t c16 = static_cast<uint16_t>(code);
  float f;
  asm("{\n\t.reg .b32 h2;\n\t.reg .b16 lo, hi;\n\t"
      "cvt.rn.f16x2.e4m3x2 h2, %1;\n\t"
      "mov.b32 {lo, hi}, h2;\n\t"
      "cvt.f32.f16 %0, lo;\n\t}"
      : "=f"(f)
      : "h"(c16));
  return f;
}

// ---------------------------------------------------------------- mbarrier + bulk copy
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but the thread may sleep up to `hint_ns` inside the instruction until the
// phase completes, instead of spinning (spinning warps take issue slots from the producer).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of parity `parity` of barrier `bar` to complete. Gives up (returns false)
// after `limit_ns`, or as soon as *abort is set when `abort` is given.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  const volatile int* abort,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  if (mbar_try_wait_sleep(bar, parity, kWaitSleepHintNs)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, kWaitSleepHintNs)) return true;
    if (abort && *abort) return false;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Bulk asynchronous copy global -> this CTA's shared memory; completion is signalled as
// `bytes` transactions on barrier `bar`. dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Prefetch `bytes` at `src` into L2 (no shared memory, no completion). Changes no memory, so it
// may run before griddepcontrol.wait: L2 is where every write becomes visible, so a line
// prefetched early can never be stale.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Programmatic dependent launch: let the next kernel of the stream be scheduled once every CTA
// of this grid got here; and block until the previous kernel of the stream has completed and
// its writes are visible (a no-op when the launch has no programmatic dependency).
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_prerequisites() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------- thread-block clusters
__device__ __forceinline__ int cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return static_cast<int>(r);
}
// The set-up cluster barrier in two halves: every thread of every CTA arrives at the start, and
// a thread's wait returns once all threads of the cluster have arrived (every CTA is running, and
// what each initialised before its arrival can be used by the others).
// The arrival has no release semantics: the barrier orders no data of its own (the exchange
// barriers' initialisation is released by fence.mbarrier_init before it).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Two floats into CTA `rank`'s copy of this CTA's shared-memory address `addr`, completing 8 bytes
// of transaction on that CTA's copy of the mbarrier at `bar`: an asynchronous store whose arrival
// the receiver sees through its barrier, with no fence on the sender's side.
__device__ __forceinline__ void st_async_f32x2(uint32_t addr, uint32_t bar, int rank, float2 v) {
  uint32_t raddr, rbar;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(raddr) : "r"(addr), "r"(rank));
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(rbar) : "r"(bar), "r"(rank));
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(
          raddr),
      "f"(v.x), "f"(v.y), "r"(rbar)
      : "memory");
}
// Split rows: the exchange of each row's (sum of squares, max) between the CTAs of a cluster.
// Every CTA holds two slot sets and two mbarriers (count 1), one of each per row parity. For a
// row of parity q, thread 0 arrives on barrier q expecting kSplit * 8 bytes, threads 0 .. kSplit-1
// push the CTA-wide pair into slot [q][own rank] of CTA 0 .. kSplit-1 (one peer each, this CTA
// included) with st.async, which completes 8 bytes on that CTA's barrier q, and every thread
// waits for the barrier's phase; then each CTA adds the kSplit pairs in rank order, so every CTA
// gets the same bits. The n-th exchanged row of a CTA uses parity n & 1 and waits on phase
// (n >> 1) & 1 of that barrier.
// Reuse: a CTA pushes into slot set q (and completes barrier q) for row n + 2 only after its own
// wait for row n + 1, which needs every CTA's push for row n + 1; a CTA pushes for row n + 1
// only after all of its threads have read the slots of row n (the row's block barrier lies in
// between) and after barrier q's phase for row n has completed. A push that arrives before the
// receiver's own arrival only makes the transaction count negative for a while.
// Start: each CTA initialises its barriers and fences the initialisation before its arrival at
// the set-up cluster barrier; the first exchange waits on that barrier first, so no CTA pushes
// into a peer that is not running or whose barriers are not ready. End: a CTA's last wait
// returns only once every push into it has landed, so it may exit right after.
// The wait is bounded (kWaitLimitNs): if it runs out (a peer stalled for seconds), the error bit
// goes to the launch's error word and the thread waits once more, with the same bound, so that a
// late push still lands in a running CTA.
__shared__ float2 g_xslots[2][8];            // this CTA's [row parity][source rank] pairs
__shared__ __align__(8) uint64_t g_xbar[2];  // this CTA's [row parity] exchange barriers

__device__ __forceinline__ void cluster_exchange_init() {
  mbar_init(smem_addr(&g_xbar[0]), 1);
  mbar_init(smem_addr(&g_xbar[1]), 1);
  fence_mbar_init();
}

template <int kSplit>
__device__ __forceinline__ float2 cluster_row_sum(float2 part, int rank, int parity,
                                                  uint32_t phase, bool& setup_seen,
                                                  unsigned int* error_word) {
  if (!setup_seen) {
    cluster_wait();
    setup_seen = true;
  }
  const uint32_t bar = smem_addr(&g_xbar[parity]);
  if (threadIdx.x == 0) mbar_arrive_expect_tx(bar, kSplit * 8u);
  if (threadIdx.x < kSplit)
    st_async_f32x2(smem_addr(&g_xslots[parity][rank]), bar, static_cast<int>(threadIdx.x), part);
  if (!mbar_wait_bounded(bar, phase, nullptr)) {
    if (threadIdx.x == 0) atomicOr(error_word, kErrWaitTimeout);
    mbar_wait_bounded(bar, phase, nullptr);
  }
  float ss = 0.0f, mx = 0.0f;
#pragma unroll
  for (int r = 0; r < kSplit; ++r) {
    const float2 v = g_xslots[parity][r];
    ss += v.x;
    mx = fmaxf(mx, v.y);
  }
  return make_float2(ss, mx);
}

// ---------------------------------------------------------------- row reduction
// Sum of squares and (optionally) max over the CTA's consumer threads, plus an OR of their abort
// votes. All consumer threads get bit-identical results (every thread adds the per-warp values
// in the same order). `slots` holds two sets of 32 per-warp slots used on alternate rows, so one
// barrier per row suffices.
template <bool kWithMax>
__device__ __forceinline__ float2 row_reduce(float ss, float mx, int abort, RedSlot* slots,
                                             int parity, int nthreads, int* abort_all) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    ss += __shfl_xor_sync(0xFFFFFFFFu, ss, o);
    if (kWithMax) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
  }
  abort = __any_sync(0xFFFFFFFFu, abort);
  const int warp = threadIdx.x >> 5;
  RedSlot* s = slots + parity * 32;
  if ((threadIdx.x & 31) == 0) {
    s[warp].ss = ss;
    s[warp].mx = mx;
    s[warp].abort = abort;
  }
  named_barrier_sync(1, nthreads);
  float tss = 0.0f, tmx = 0.0f;
  int ab = 0;
  for (int w = 0; w < (nthreads >> 5); ++w) {
    const float4 slot = *reinterpret_cast<const float4*>(&s[w]);  // one 16-byte load
    tss += slot.x;
    if (kWithMax) tmx = fmaxf(tmx, slot.y);
    ab |= __float_as_int(slot.z);
  }
  *abort_all = ab;
  return make_float2(tss, tmx);
}

// ---------------------------------------------------------------- per-row epilogue
// Constants of the quantiser, read once per thread.
struct QuantConst {
  float inv_scale;  // FP8 static: 1 / scale
  float gs;         // NVFP4: global (encode) scale
};

template <int kMode>
__device__ __forceinline__ QuantConst load_quant_const(const Params& p) {
  QuantConst q{0.0f, 0.0f};
  if (kMode == kModeFp8Static) q.inv_scale = 1.0f / __ldg(p.scale);
  if (kMode == kModeNvfp4) q.gs = __ldg(p.scale);
  return q;
}

// Byte offset of NVFP4 block scale (row t, block b): row-major [T_pad][H/16], or the 128x4-tile
// layout block-scaled GEMMs read (scale matrix padded to 128 rows x 4 columns; tile (i, j) is a
// 512-byte block at (i * sf_cols/4 + j) * 512, row r / column c of it at (r%32)*16 + (r/32)*4 + c).
// Split as a per-row base (computed once per row) plus a per-block column offset.
__device__ __forceinline__ int64_t scale_row_base(const Params& p, int64_t t) {
  if (!p.scale_swizzled) return t * (p.H / 16);
  const int r = static_cast<int>(t & 127);
  return (t >> 7) * static_cast<int64_t>(p.sf_cols) * 128 + (r & 31) * 16 + (r >> 5) * 4;
}
__device__ __forceinline__ int scale_col_offset(const Params& p, int b) {
  return p.scale_swizzled ? (b >> 2) * 512 + (b & 3) : b;
}
__device__ __forceinline__ int64_t scale_offset(const Params& p, int64_t t, int b) {
  return scale_row_base(p, t) + scale_col_offset(p, b);
}

// Swizzled layout: the padding columns H/16 .. sf_cols of a row (at most 3) are zero. Block
// column b pairs with vectors 2b, 2b+1; the thread that owns vector v = 2b (v >= nvec for a
// padding column) writes the zero. Threads cover nthreads*VEC >= nvec rounded up to 32*VEC
// vectors, which reaches 2*sf_cols (nvec rounded up to 8).
__device__ __forceinline__ bool is_scale_pad_vector(const Params& p, int v) {
  return p.scale_swizzled && v >= p.nvec && (v & 1) == 0 && v < 2 * p.sf_cols;
}

// Split rows: the swizzled layout's padding scale columns of row t, written by thread 0 of the
// cluster's first CTA.
__device__ __forceinline__ void zero_scale_pad_columns(const Params& p, int64_t t, int c,
                                                       int vbase) {
  if (!p.scale_swizzled || c != 0 || vbase != 0) return;
  uint8_t* sf_row = static_cast<uint8_t*>(p.out_scales) + scale_row_base(p, t);
  for (int b = p.H / 16; b < p.sf_cols; ++b) sf_row[scale_col_offset(p, b)] = 0;
}

// Zero every output byte of padding row t that this thread owns. Rows at or beyond T_pad exist
// only in the swizzled NVFP4 scale layout (rows padded to 128): there only the scales are written.
// Split rows (kSplit > 1): this CTA owns vectors [vbase, vend) of the row.
template <int kVec, int kMode, int kSplit = 1>
__device__ __forceinline__ void zero_row(const Params& p, int64_t t, int c, int vbase = 0,
                                         int vend = 0) {
  const int64_t H = p.H;
  const bool real_row = t < p.T_pad;
#pragma unroll
  for (int k = 0; k < kVec; ++k) {
    const int v = (kSplit > 1 ? vbase : 0) + c + k * p.nthreads;
    if (kMode == kModeNvfp4 && kSplit == 1 && is_scale_pad_vector(p, v))
      static_cast<uint8_t*>(p.out_scales)[scale_offset(p, t, v / 2)] = 0;
    if (v >= (kSplit > 1 ? vend : p.nvec)) continue;
    if (real_row) stg_stream(p.residual_out + t * H + v * 8, make_uint4(0, 0, 0, 0));
    if (kMode != kModeNvfp4 && !real_row) continue;
    if (kMode == kModeNone) {
      stg_stream(static_cast<uint16_t*>(p.out) + t * H + v * 8, make_uint4(0, 0, 0, 0));
    } else if (kMode == kModeFp8Static || kMode == kModeFp8PerToken) {
      stg_stream(static_cast<uint8_t*>(p.out) + t * H + v * 8, make_uint2(0, 0));
    } else {
      if (real_row) stg_stream(static_cast<uint8_t*>(p.out) + t * (H / 2) + v * 4, 0u);
      if ((v & 1) == 0) static_cast<uint8_t*>(p.out_scales)[scale_offset(p, t, v / 2)] = 0;
    }
  }
  if (kMode == kModeFp8PerToken && c == 0 && (kSplit == 1 || vbase == 0) && real_row)
    static_cast<float*>(p.out_scales)[t] = 0.0f;
  if (kMode == kModeNvfp4 && kSplit > 1) zero_scale_pad_columns(p, t, c, vbase);
}

// Finish row t: h holds sum_r partials + residual + bias for this thread's vectors (zero for
// vectors past the row). Writes residual_out, normalises, quantises and stores. Returns the
// CTA-wide abort vote. Split rows (kSplit > 1): this CTA (cluster rank `rank`) owns vectors
// [vbase, vend) and the row's sums are combined across the cluster by cluster_row_sum.
template <int kVec, int kMode, int kSplit = 1>
__device__ __forceinline__ int finish_row(const Params& p, int64_t t, float (&h)[kVec][8],
                                          const uint4 (&w)[kVec], const QuantConst& qc,
                                          RedSlot* slots, int parity, int c, int abort,
                                          int vbase = 0, int vend = 0, int rank = 0,
                                          bool* setup_seen = nullptr, uint32_t xphase = 0) {
  const int64_t H = p.H;
  const int v0 = kSplit > 1 ? vbase : 0;
  const int vlim = kSplit > 1 ? vend : p.nvec;
  float ss0 = 0.0f, ss1 = 0.0f;  // sums of squares of the even and the odd elements
  // Split rows: the new residual is stored after the exchange (storing it before measured the
  // same to 1.5 % slower on decode calls, GB300 A/B).
  uint4 res[kSplit > 1 ? kVec : 1];
#pragma unroll
  for (int k = 0; k < kVec; ++k) {
    const int v = v0 + c + k * p.nthreads;
    if constexpr (kSplit > 1)
      res[k] = pack_bf16x8(h[k]);
    else if (v < vlim)
      stg_stream(p.residual_out + t * H + v * 8, pack_bf16x8(h[k]));
#pragma unroll
    for (int e = 0; e < 8; e += 2) fma2(ss0, ss1, h[k][e], h[k][e + 1], h[k][e], h[k][e + 1]);
  }
  const float ss = ss0 + ss1;
  // h <- h * w (the weight is applied before the common factor 1/rms)
  float mx = 0.0f;
#pragma unroll
  for (int k = 0; k < kVec; ++k) {
    float wf[8];
    unpack_bf16x8(w[k], wf);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      h[k][e] *= wf[e];
      if (kMode == kModeFp8PerToken) mx = fmaxf(mx, fabsf(h[k][e]));
    }
  }
  int abort_all = 0;
  float2 red =
      row_reduce<kMode == kModeFp8PerToken>(ss, mx, abort, slots, parity, p.nthreads, &abort_all);
  if constexpr (kSplit > 1) {
    red = cluster_row_sum<kSplit>(red, rank, parity, xphase, *setup_seen, p.error_word);
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int v = v0 + c + k * p.nthreads;
      if (v < vlim) stg_stream(p.residual_out + t * H + v * 8, res[k]);
    }
  }
  const float rinv = rsqrtf(red.x / static_cast<float>(p.H) + p.eps);

  if (kMode == kModeNone) {
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int v = v0 + c + k * p.nthreads;
      scale8(h[k], rinv);
      if (v < vlim) stg_stream(static_cast<uint16_t*>(p.out) + t * H + v * 8, pack_bf16x8(h[k]));
    }
  } else if (kMode == kModeFp8Static) {
    const float rinv_q = rinv * qc.inv_scale;  // y / scale = h*w * (rinv / scale)
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int v = v0 + c + k * p.nthreads;
      float* q = h[k];
      scale8(h[k], rinv_q);
      if (v < vlim)
        stg_stream(static_cast<uint8_t*>(p.out) + t * H + v * 8,
                   make_uint2(pack_e4m3x4(q[0], q[1], q[2], q[3]),
                              pack_e4m3x4(q[4], q[5], q[6], q[7])));
    }
  } else if (kMode == kModeFp8PerToken) {
    // s_t = max|y| / 448 with max|y| = max|h*w| * rinv; the codes are y / s_t = h*w * 448/max|h*w|
    const float mxhw = red.y;
    const float s = (mxhw * rinv) / 448.0f;
    if (c == 0 && v0 == 0) static_cast<float*>(p.out_scales)[t] = s;
    float f = 448.0f / mxhw;
    const bool by_division = !(f <= 3.0e38f);  // max|h*w| is zero or tiny
    if (s == 0.0f) f = 0.0f;
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int v = v0 + c + k * p.nthreads;
      float q[8];
#pragma unroll
      for (int e = 0; e < 8; ++e)
        q[e] = (by_division && s != 0.0f) ? __fdiv_rn(h[k][e], mxhw) * 448.0f : h[k][e] * f;
      if (v < vlim)
        stg_stream(static_cast<uint8_t*>(p.out) + t * H + v * 8,
                   make_uint2(pack_e4m3x4(q[0], q[1], q[2], q[3]),
                              pack_e4m3x4(q[4], q[5], q[6], q[7])));
    }
  } else {  // NVFP4: 16-element blocks = vectors (2m, 2m+1), held by lanes (c, c^1)
    uint8_t* sf_row = static_cast<uint8_t*>(p.out_scales) + scale_row_base(p, t);
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int v = v0 + c + k * p.nthreads;
      float y[8];
      float amax = 0.0f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        y[e] = h[k][e] * rinv;
        amax = fmaxf(amax, fabsf(y[e]));
      }
      amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
      const uint32_t sf = e4m3_code((amax * qc.gs) / 6.0f);
      const float sfv = e4m3_value(sf);
      const float mult = sfv == 0.0f ? 0.0f : qc.gs / sfv;
#pragma unroll
      for (int e = 0; e < 8; ++e) y[e] *= mult;
      if (v < vlim) {
        stg_stream(static_cast<uint8_t*>(p.out) + t * (H / 2) + v * 4, pack_e2m1x8(y));
        if ((v & 1) == 0) sf_row[scale_col_offset(p, v >> 1)] = static_cast<uint8_t>(sf);
      } else if (kSplit == 1 && is_scale_pad_vector(p, v)) {
        sf_row[scale_col_offset(p, v >> 1)] = 0;
      }
    }
    if (kSplit > 1) zero_scale_pad_columns(p, t, c, v0);
  }
  return abort_all;
}

// This thread's weight and bias vectors (zero past the row).
template <int kVec, int kSplit = 1>
__device__ __forceinline__ void load_row_constants(const Params& p, int c, uint4 (&w)[kVec],
                                                   uint4 (&b)[kVec], int vbase = 0,
                                                   int vend = 0) {
#pragma unroll
  for (int k = 0; k < kVec; ++k) {
    const int v = (kSplit > 1 ? vbase : 0) + c + k * p.nthreads;
    const bool ok = v < (kSplit > 1 ? vend : p.nvec);
    w[k] = ok ? ldg_keep(p.weight + v * 8) : make_uint4(0, 0, 0, 0);
    b[k] = (ok && p.bias) ? ldg_keep(p.bias + v * 8) : make_uint4(0, 0, 0, 0);
  }
}

}  // namespace spk
