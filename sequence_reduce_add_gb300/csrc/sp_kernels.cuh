// sp_kernels.cuh — the two kernels of the fused stage. Both map one token row at a time to one
// CTA, or to one cluster of CTAs in k_direct's split variant (rows are independent: RMSNorm and
// every scale kind used here are per token), walk rows
// in token order (a grid stride, or claimed in the staged kernel's dynamic variant below), and
// make a single pass over HBM: every partial, residual and output byte of a valid row is read
// or written exactly once; padding rows are written as zeros without any read.
//
// Thread c of the CTA's consumer threads owns 16-byte vectors v = c + k*nthreads (k < VEC) of
// the row, i.e. 8*VEC columns, held as fp32 accumulators in registers for the whole row.
//
//   k_staged  A producer thread streams the row's tp partial rows, its residual row and its
//             addend row (each a contiguous 2*H-byte segment) into a ring of stages with bulk
//             asynchronous copies (cp.async.bulk, completion on an mbarrier per stage) while the
//             consumer warps add the segments that have landed. The ring runs ahead across rows,
//             so HBM stays busy through each row's reduction and epilogue, and the bytes in flight
//             per SM are set by the ring depth rather than by registers.
//             Rows go to CTAs either statically (CTA b takes rows b, b + grid, ...) or, in the
//             dynamic variant, as claimed: CTA b starts with row b and then claims rows from a
//             per-stream counter one row ahead, so CTAs that get more bandwidth take more rows and
//             all finish within about one row of each other. The producer passes each row's index
//             to the consumers beside the row's first ring stage.
//   k_direct  The consumer threads load their vectors of every segment straight into registers
//             with 128-bit non-coherent loads: the residual row first, then the partials four or
//             eight rows at a time. Its split variant shares each row among the CTAs of a
//             thread-block cluster, each owning a contiguous slice, for calls with few rows.
#pragma once

#include "sp_device.cuh"

namespace spk {

constexpr int kMaxConsumerThreads = 512;  // 16 warps
constexpr int kProducerThreads = 32;

// Row counters of the dynamic schedule: slot i is [next claim, CTAs done]. A launch gets the
// address of one pair (a slot of this table chosen by its stream, or a caller's own pair); its
// last CTA to finish claiming sets both words back to zero, so the next launch using that pair
// (which starts claiming only after this one has completed) finds it zeroed.
constexpr int kRowCounterSlots = 256;
__device__ unsigned int g_row_counters[2 * kRowCounterSlots];
// Per slot, the sequence number of the last launch on it that has reset it (written by that
// launch's last CTA to finish claiming, after the reset). The host compares it with the number of
// launches it issued on the slot to tell when the slot is idle and may go to another stream.
__device__ unsigned long long g_row_counter_done[kRowCounterSlots];

// The CTA's error word address, kept in shared memory beside the abort flag: a report site (a
// cold path inside the row loops) reads it there instead of holding it in registers.
__device__ __forceinline__ unsigned int* error_word_of(int* abort_flag) {
  return *reinterpret_cast<unsigned int* volatile*>(abort_flag + 2);
}

// ----------------------------------------------------------------------------------- staged
// kTest: the self-test instantiation (sp_selftest_fused_timeout): every bounded wait uses the
// launch's p.wait_limit_ns and CTA 0's producer withholds ring fill number p.withhold. Production
// instantiations use the fixed limit and withhold nothing.
template <int kVec, int kMode, bool kDynamic, bool kTest = false>
__global__ void __launch_bounds__(kMaxConsumerThreads + kProducerThreads)
    k_staged(const Params p) {
  const uint64_t wait_limit = kTest ? p.wait_limit_ns : kWaitLimitNs;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + p.stages;
  RedSlot* slots = reinterpret_cast<RedSlot*>(empty + p.stages);
  int* abort_flag = reinterpret_cast<int*>(slots + 64);
  int64_t* row_ids = reinterpret_cast<int64_t*>(abort_flag + 4);  // [stages], dynamic schedule
  unsigned char* ring = smem + p.ring_offset;

  const int tid = threadIdx.x;
  const int nc = p.nthreads;
  // Row segments in stream order: partials 0 .. tp-1, then residual, then addend (if present).
  const int nseg = p.tp + (p.residual ? 1 : 0) + (p.addend ? 1 : 0);
  auto segment = [&](int64_t t, int seg) -> const uint16_t* {
    if (seg < p.tp) return p.partials + seg * p.plane + t * static_cast<int64_t>(p.H);
    if (seg == p.tp && p.residual) return p.residual + t * static_cast<int64_t>(p.H);
    return p.addend + t * static_cast<int64_t>(p.H);
  };
  const uint32_t seg_bytes = static_cast<uint32_t>(p.H) * 2u;

  if (tid == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(smem_addr(full + s), 1);
      mbar_init(smem_addr(empty + s), static_cast<uint32_t>(nc >> 5));
    }
    *abort_flag = 0;
    *reinterpret_cast<unsigned int**>(abort_flag + 2) = p.error_word;
    fence_mbar_init();
  } else if (tid == nc) {
    // While the previous kernel of the stream may still be running, pull this CTA's first ring
    // of segments, and the weight and bias, into L2 so that the first reads after the wait hit L2.
    bulk_prefetch_l2(p.weight, seg_bytes);
    if (p.bias) bulk_prefetch_l2(p.bias, seg_bytes);
    int n = 0;
    for (int64_t t = blockIdx.x; t < p.T_valid && n < p.stages; t += gridDim.x)
      for (int seg = 0; seg < nseg && n < p.stages; ++seg, ++n)
        bulk_prefetch_l2(segment(t, seg), seg_bytes);
  }
  pdl_launch_dependents();
  pdl_wait_prerequisites();
  __syncthreads();

  if (tid >= nc) {
    // ------------------------------------------------------------ producer (one thread)
    if (tid != nc) return;
    const uint64_t policy = l2_evict_first_policy();
    const int64_t withhold = (kTest && blockIdx.x == 0) ? p.withhold : -1;
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    bool aborted = false;
    if constexpr (!kDynamic) {
      for (int64_t t = blockIdx.x; t < p.T_valid && !aborted; t += gridDim.x) {
        for (int seg = 0; seg < nseg; ++seg) {
          const uint16_t* src = segment(t, seg);
          if (!mbar_wait_bounded(smem_addr(empty + stage), phase ^ 1u, abort_flag,
                                 wait_limit)) {
            if (!*static_cast<volatile int*>(abort_flag))
            atomicOr(error_word_of(abort_flag), kErrWaitTimeout);
            *static_cast<volatile int*>(abort_flag) = 1;
            aborted = true;
            break;
          }
          if (kTest && issued == withhold) {  // this stage never fills; issue nothing more
            ++issued;
            aborted = true;
            break;
          }
          const uint32_t bar = smem_addr(full + stage);
          mbar_arrive_expect_tx(bar, seg_bytes);
          bulk_g2s(smem_addr(ring + stage * p.seg_stride), src, seg_bytes, bar, policy);
          ++issued;
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    } else {
      // Every row, padding rows included, takes one ring stage for its index (a padding row and
      // the final -1 take it alone: the producer completes that stage's phase by arriving).
      unsigned int* counter = p.row_counter;
      int64_t next = blockIdx.x;
      for (;;) {
        const int64_t t = next < p.rows_total ? next : -1;
        if (t >= 0) next = static_cast<int64_t>(gridDim.x) + atomicAdd(counter, 1u);
        for (int seg = 0; seg < (t >= 0 && t < p.T_valid ? nseg : 1); ++seg) {
          if (!mbar_wait_bounded(smem_addr(empty + stage), phase ^ 1u, abort_flag,
                                 wait_limit)) {
            if (!*static_cast<volatile int*>(abort_flag))
            atomicOr(error_word_of(abort_flag), kErrWaitTimeout);
            *static_cast<volatile int*>(abort_flag) = 1;
            aborted = true;
            break;
          }
          const uint32_t bar = smem_addr(full + stage);
          if (seg == 0) row_ids[stage] = t;
          if (kTest && issued == withhold) {  // this stage never fills; issue nothing more
            ++issued;
            aborted = true;
            break;
          }
          if (t >= 0 && t < p.T_valid) {
            mbar_arrive_expect_tx(bar, seg_bytes);
            bulk_g2s(smem_addr(ring + stage * p.seg_stride), segment(t, seg), seg_bytes, bar,
                     policy);
          } else {
            mbar_arrive(bar);
          }
          ++issued;
          if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (aborted || t < 0) break;
      }
    }
    // Let every copy still in flight land before this CTA can exit: wait for the last issued
    // phase of each stage.
    const int64_t used = issued < p.stages ? issued : p.stages;
    for (int64_t s = 0; s < used; ++s) {
      const int64_t last = issued - 1 - ((issued - 1 - s) % p.stages);  // last issue on stage s
      const uint32_t par = static_cast<uint32_t>((last / p.stages) & 1);
      if (!mbar_wait_bounded(smem_addr(full + s), par, nullptr, wait_limit))
        atomicOr(error_word_of(abort_flag), kErrWaitTimeout);
    }
    if constexpr (kDynamic) {
      // This CTA claims no more rows; the last CTA of the launch to get here resets the pair.
      unsigned int* counter = p.row_counter;
      __threadfence();
      if (atomicAdd(counter + 1, 1u) == gridDim.x - 1) {
        counter[0] = 0u;
        counter[1] = 0u;
        __threadfence();
        if (p.slot_done) *reinterpret_cast<volatile unsigned long long*>(p.slot_done) = p.slot_seq;
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int c = tid;
  const int lane = tid & 31;
  // This thread's weight and bias vectors live in shared memory (read once per row) rather than
  // in registers, so that more rows fit on an SM. Each thread writes and reads only its own
  // vectors, so no barrier is needed.
  uint4* wb = reinterpret_cast<uint4*>(smem + p.wb_offset);
  {
    uint4 w0[kVec], b0[kVec];
    load_row_constants<kVec>(p, c, w0, b0);
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int v = c + k * nc;
      if (v < p.nvec) {
        wb[v] = w0[k];
        wb[p.nvec + v] = b0[k];
      }
    }
  }
  const QuantConst qc = load_quant_const<kMode>(p);

  int stage = 0;
  uint32_t phase = 0;
  int parity = 0;
  for (int64_t t_static = blockIdx.x;; t_static += gridDim.x) {
    int64_t t = t_static;
    if constexpr (!kDynamic) {
      if (t >= p.rows_total) break;
      if (t >= p.T_valid) {
        zero_row<kVec, kMode>(p, t, c);
        continue;
      }
    } else {
      // The row's index sits beside its first stage. A warp acts on the wait only as a whole.
      // Every warp leaves the loop through exactly one row barrier after the last one all warps
      // passed together: the abort vote here (a warp whose wait ran out), the bare barrier below
      // (no more rows), or a row's own barrier in finish_row. All warps read the same row
      // indices, so whatever mix of these the warps take, each takes one; warps at a row's
      // barrier then read the abort vote and leave too. (Leaving without a barrier on "no more
      // rows" could strand a sibling warp in its abort vote if its wait ran out just as the
      // stage completed.)
      const bool landed =
          mbar_wait_bounded(smem_addr(full + stage), phase, abort_flag, wait_limit);
      if (!__all_sync(0xFFFFFFFFu, landed)) {
        if (lane == 0) {
          if (!*static_cast<volatile int*>(abort_flag))
            atomicOr(error_word_of(abort_flag), kErrWaitTimeout);
          *static_cast<volatile int*>(abort_flag) = 1;
        }
        int ignored = 0;
        row_reduce<false>(0.0f, 0.0f, 1, slots, parity, nc, &ignored);
        break;
      }
      t = row_ids[stage];
      if (t < 0) {
        named_barrier_sync(1, nc);
        break;
      }
      if (t >= p.T_valid) {
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(empty + stage));
        if (++stage == p.stages) {
          stage = 0;
          phase ^= 1u;
        }
        zero_row<kVec, kMode>(p, t, c);
        continue;
      }
    }
    // The accumulator starts from the bias (zero without one), which keeps that load off the
    // row epilogue's critical path; with a partial scale the bias joins after the scaling.
    // Not for per-token FP8: there the earlier load costs a register spill (measured 3 % slower
    // at tp=16, H=8192), while NVFP4 gains 1.5 % and bf16 / static FP8 are unchanged.
    const bool bias_first = kMode != kModeFp8PerToken && p.partial_scale == 1.0f;
    float h[kVec][8];
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int v = c + k * nc;
      unpack_bf16x8(bias_first && v < p.nvec ? wb[p.nvec + v] : make_uint4(0, 0, 0, 0), h[k]);
    }

    int aborted = 0;
    for (int seg = 0; seg < nseg; ++seg) {
      if (!aborted &&
          !mbar_wait_bounded(smem_addr(full + stage), phase, abort_flag, wait_limit)) {
        if (!*static_cast<volatile int*>(abort_flag))
          atomicOr(error_word_of(abort_flag), kErrWaitTimeout);
        *static_cast<volatile int*>(abort_flag) = 1;
        aborted = 1;
      }
      const unsigned char* src = ring + stage * p.seg_stride;
#pragma unroll
      for (int k = 0; k < kVec; ++k) {
        const int v = c + k * nc;
        if (v < p.nvec) add_bf16x8(*reinterpret_cast<const uint4*>(src + v * 16), h[k]);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(empty + stage));
      if (++stage == p.stages) {
        stage = 0;
        phase ^= 1u;
      }
      if (seg + 1 == p.tp && !bias_first) {  // the reduced partial sum is complete: scale it
#pragma unroll
        for (int k = 0; k < kVec; ++k) {
          const int v = c + k * nc;
          scale8(h[k], p.partial_scale);
          if (v < p.nvec) add_bf16x8(wb[p.nvec + v], h[k]);
        }
      }
    }
    uint4 w[kVec];
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int v = c + k * nc;
      w[k] = v < p.nvec ? wb[v] : make_uint4(0, 0, 0, 0);
    }
    const int stop = finish_row<kVec, kMode>(p, t, h, w, qc, slots, parity, c, aborted);
    parity ^= 1;
    if (stop) break;  // every consumer sees the same vote, so all leave together
  }
  // A consumer whose wait ran out set the abort flag before the row barrier that every
  // consumer passed on the way out, so thread 0 sees it here and reports it once for the CTA.

}

// ----------------------------------------------------------------------------------- direct
// kSplit > 1: each row is split across the kSplit CTAs of a thread-block cluster, CTA r owning
// vectors [r * split_chunk, (r + 1) * split_chunk) of it; the CTAs combine the row's sum of
// squares (and max) through distributed shared memory. A call with few rows then draws on
// kSplit times as many SMs.
// kBatch: partial rows whose loads are in flight together (4, or 8 with one vector per thread:
// more in flight per row, about twice the registers).
template <int kVec, int kMode, int kSplit, int kBatch>
__global__ void __launch_bounds__(kMaxConsumerThreads) k_direct(const Params p) {
  static_assert(kBatch == 4 || (kBatch == 8 && kVec == 1), "batch of 4, or 8 at one vector");
  constexpr bool kEarlyResidual = kVec <= 2;  // residual row loaded before the partials
  __shared__ RedSlot slots[64];
  const int c = threadIdx.x;
  const int nc = p.nthreads;
  const int64_t H = p.H;
  const int rank = kSplit > 1 ? cluster_rank() : 0;
  const int vbase = kSplit > 1 ? rank * p.split_chunk : 0;
  const int vend = kSplit > 1 ? min(vbase + p.split_chunk, p.nvec) : p.nvec;
  const int vc = vbase + c;  // this thread's first vector
  bool setup_seen = false;  // split rows: waited on the set-up cluster barrier
  // split rows: the exchange barriers, then the set-up cluster barrier (cluster_row_sum)
  if constexpr (kSplit > 1) {
    if (c == 0) cluster_exchange_init();
    cluster_arrive_relaxed();
  }
  pdl_wait_prerequisites();
  uint4 w[kVec], b[kVec];
  load_row_constants<kVec, kSplit>(p, c, w, b, vbase, vend);
  const QuantConst qc = load_quant_const<kMode>(p);

  // rows finished so far (padding rows aside): the row's parity is its low bit, and for split
  // rows the phase of the exchange barrier it waits on is the next bit
  unsigned done = 0;
  // every CTA of a cluster takes the same rows, so all take part in the same exchanges
  for (int64_t t = blockIdx.x / kSplit; t < p.rows_total; t += gridDim.x / kSplit) {
    if (t >= p.T_valid) {
      zero_row<kVec, kMode, kSplit>(p, t, c, vbase, vend);
      continue;
    }
    float h[kVec][8];
#pragma unroll
    for (int k = 0; k < kVec; ++k)
#pragma unroll
      for (int e = 0; e < 8; ++e) h[k][e] = 0.0f;

    // The residual row's loads go out first, then the partials' kBatch rows at a time (every
    // batch full width, the missing rows predicated off), so a row costs about one round trip to
    // memory per batch.
    uint4 xres[kVec];
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const int v = vc + k * nc;
      xres[k] = (kEarlyResidual && p.residual && v < vend) ? ldg_stream(p.residual + t * H + v * 8)
                                                           : make_uint4(0, 0, 0, 0);
    }
    const uint16_t* row = p.partials + t * H;
    int r = 0;
    if constexpr (kVec <= 2) {
#pragma unroll 1
      for (; r < p.tp; r += kBatch) {
        uint4 x[kBatch][kVec];
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
#pragma unroll
          for (int k = 0; k < kVec; ++k) {
            const int v = vc + k * nc;
            x[u][k] = (r + u < p.tp && v < vend) ? ldg_stream(row + (r + u) * p.plane + v * 8)
                                                 : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
          if (r + u < p.tp) {
#pragma unroll
            for (int k = 0; k < kVec; ++k) add_bf16x8(x[u][k], h[k]);
          }
      }
    } else {  // four vectors per thread: full batches, then the rest one row at a time
      for (; r + kBatch <= p.tp; r += kBatch) {
        uint4 x[kBatch][kVec];
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
#pragma unroll
          for (int k = 0; k < kVec; ++k) {
            const int v = vc + k * nc;
            x[u][k] = v < vend ? ldg_stream(row + (r + u) * p.plane + v * 8) : make_uint4(0, 0, 0, 0);
          }
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
#pragma unroll
          for (int k = 0; k < kVec; ++k) add_bf16x8(x[u][k], h[k]);
      }
      for (; r < p.tp; ++r) {
#pragma unroll
        for (int k = 0; k < kVec; ++k) {
          const int v = vc + k * nc;
          if (v < vend) add_bf16x8(ldg_stream(row + r * p.plane + v * 8), h[k]);
        }
      }
    }
    if (p.partial_scale != 1.0f) {
#pragma unroll
      for (int k = 0; k < kVec; ++k) scale8(h[k], p.partial_scale);
    }
    if (p.residual) {
#pragma unroll
      for (int k = 0; k < kVec; ++k) {
        const int v = vc + k * nc;
        if (kEarlyResidual)
          add_bf16x8(xres[k], h[k]);
        else if (v < vend)
          add_bf16x8(ldg_stream(p.residual + t * H + v * 8), h[k]);
      }
    }
    if (p.addend) {
#pragma unroll
      for (int k = 0; k < kVec; ++k) {
        const int v = vc + k * nc;
        if (v < vend) add_bf16x8(ldg_stream(p.addend + t * H + v * 8), h[k]);
      }
    }
#pragma unroll
    for (int k = 0; k < kVec; ++k) add_bf16x8(b[k], h[k]);
    finish_row<kVec, kMode, kSplit>(p, t, h, w, qc, slots, static_cast<int>(done & 1u), c, 0,
                                    vbase, vend, rank, &setup_seen, (done >> 1) & 1u);
    ++done;
  }
  // A CTA that made no exchange still completes the set-up barrier it arrived at.
  if constexpr (kSplit > 1) {
    if (!setup_seen) cluster_wait();
  }
  // The next kernel of the stream is let in only now, at the end (an exit would do the same):
  // letting it in at the start, so that its CTAs wait beside these ones, measured 5-15 % slower
  // on calls of up to a few hundred rows (GB300 A/B, back to back).
  pdl_launch_dependents();
}

// ------------------------------------------------------------------------------------ slice
// The staged kernel's split-row form: one row per cluster of kSplit CTAs (cluster b takes row
// b), CTA r owning vectors [r * split_chunk, (r + 1) * split_chunk) of the row as in k_direct's
// split variant. The CTA brings its slice of every segment of the row (the tp partials, the
// residual, the addend) into shared memory with one bulk asynchronous copy each, all in flight at
// once and none held in registers, then adds them, and the cluster combines the row's sums as
// k_direct's split rows do (cluster_row_sum). A call whose rows' slices all fit on the SMs at once
// then costs one round trip to memory per row and draws on every SM.
template <int kMode, int kSplit>
__global__ void __launch_bounds__(kMaxConsumerThreads) k_slice(const Params p) {
  static_assert(kSplit >= 2 && kSplit <= 8, "a cluster of 2 to 8 CTAs per row");
  extern __shared__ __align__(128) unsigned char smem[];  // [segment][slice vector] uint4
  __shared__ RedSlot slots[64];
  __shared__ __align__(8) uint64_t loaded;
  const int c = threadIdx.x;
  const int64_t H = p.H;
  const int rank = cluster_rank();
  const int vbase = rank * p.split_chunk;
  const int vend = min(vbase + p.split_chunk, p.nvec);
  const int nv = vend > vbase ? vend - vbase : 0;  // this CTA's vectors of the row
  const int64_t t = blockIdx.x / kSplit;
  bool setup_seen = false;
  if (c == 0) {
    cluster_exchange_init();
    mbar_init(smem_addr(&loaded), 1);
    fence_mbar_init();
  }
  cluster_arrive_relaxed();
  __syncthreads();
  pdl_wait_prerequisites();
  if (t >= p.T_valid) {  // a padding row (or a row past T_pad of the swizzled scale layout)
    zero_row<1, kMode, kSplit>(p, t, c, vbase, vend);
    cluster_wait();  // complete the set-up barrier this CTA arrived at
    pdl_launch_dependents();
    return;
  }
  const int nseg = p.tp + (p.residual ? 1 : 0) + (p.addend ? 1 : 0);
  const uint32_t bar = smem_addr(&loaded);
  if (c < 32) {
    if (c == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nseg * nv) * 16u);
    if (nv > 0) {
      const uint64_t policy = l2_evict_first_policy();
      for (int seg = c; seg < nseg; seg += 32) {
        const uint16_t* row = seg < p.tp                     ? p.partials + seg * p.plane
                            : (seg == p.tp && p.residual) ? p.residual
                                                          : p.addend;
        bulk_g2s(smem_addr(smem + static_cast<size_t>(seg) * nv * 16), row + t * H + vbase * 8,
                 static_cast<uint32_t>(nv) * 16u, bar, policy);
      }
    }
  }
  uint4 w[1], b[1];
  load_row_constants<1, kSplit>(p, c, w, b, vbase, vend);
  const QuantConst qc = load_quant_const<kMode>(p);
  if (!mbar_wait_bounded(bar, 0, nullptr)) {
    if (c == 0) atomicOr(p.error_word, kErrWaitTimeout);
    mbar_wait_bounded(bar, 0, nullptr);  // let the copies land before the CTA goes on
  }
  float h[1][8];
#pragma unroll
  for (int e = 0; e < 8; ++e) h[0][e] = 0.0f;
  if (c < nv) {
    const uint4* seg0 = reinterpret_cast<const uint4*>(smem) + c;
    for (int r = 0; r < p.tp; ++r) add_bf16x8(seg0[r * nv], h[0]);
    if (p.partial_scale != 1.0f) scale8(h[0], p.partial_scale);
    int seg = p.tp;
    if (p.residual) add_bf16x8(seg0[seg++ * nv], h[0]);
    if (p.addend) add_bf16x8(seg0[seg * nv], h[0]);
  }
  add_bf16x8(b[0], h[0]);
  finish_row<1, kMode, kSplit>(p, t, h, w, qc, slots, 0, c, 0, vbase, vend, rank, &setup_seen, 0);
  pdl_launch_dependents();  // only at the end, as in k_direct (early: up to 37 % slower)
}

// ----------------------------------------------------------------------------------- self-test
// The timeout path of the bounded waits, on the GPU: one warp waits, with the given limit, on an
// mbarrier that nothing arrives at. The wait must give up, record SP_DEVICE_ERR_WAIT_TIMEOUT in
// the device error word and let the kernel finish normally.
__global__ void k_selftest_wait_timeout(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  const bool done = mbar_wait_bounded(smem_addr(&bar), 0, nullptr, limit_ns);
  if (!done && threadIdx.x == 0) atomicOr(&g_error_flags, kErrWaitTimeout);
}

}  // namespace spk
