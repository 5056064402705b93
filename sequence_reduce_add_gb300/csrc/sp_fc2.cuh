// sp_fc2.cuh — FlashComm2 token reorganisation on one GPU (vllm-ascend SP/FlashComm notes
// §4.2-4.4): all G = global_tp ranks' [N][H/G] feature slices live in one buffer x [G][N][F]
// (F = H/G); the output y [G][N/D][D*F] (D = odp_size = G/P, P = otp_size) is what every rank
// holds after the local reorder by the reorganised batch ids, the ODP-group all_to_all and the
// feature concat.
//
// Closed form of that map: output rank r = g*D + j, output row i = k*S + tl (S = N/G tokens
// per segment, k < P, tl < S), feature block m < D  <-  source rank g*D + m, source token
// (j + k*D)*S + tl, all F features. Each such (r, i, m) piece is F contiguous elements on both
// sides; pieces are numbered in output order, so the writes stream sequentially.
//
//   k_fc2_bulk        A tile is a run of consecutive output pieces. One warp per CTA gathers a
//                     tile's pieces into shared memory with one bulk copy each (in output order),
//                     then writes the tile back with a single bulk store; a ring of tiles keeps
//                     loads in flight while earlier tiles drain.
//   k_fc2_reorganize  One warp per piece through registers; used when one piece is larger than
//                     a ring stage.
#pragma once

#include "sp_device.cuh"

namespace spk {

// Bulk asynchronous copy this CTA's shared memory -> global, tracked in the issuing thread's
// bulk group. dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_s2g(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Block until at most kPending of this thread's committed bulk groups are still reading their
// shared-memory source.
template <int kPending>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(kPending) : "memory");
}
// Block until every committed bulk group of this thread has completed (writes performed).
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Order this thread's earlier shared-memory accesses before its later async-proxy operations.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

struct Fc2Params {
  const unsigned char* x;
  unsigned char* y;
  int64_t N;           // tokens
  int64_t pieces;      // G * N: pieces of F elements
  int64_t S;           // tokens per segment, N / G
  int D;               // odp_size
  int P;               // otp_size
  int piece_vecs;      // F * elem_bytes / 16
  // k_fc2_bulk only
  uint32_t piece_bytes;  // F * elem_bytes
  int tile_pieces;       // pieces per tile (one ring stage)
  int stages;            // ring depth (<= kFc2MaxStages)
  uint32_t stage_bytes;  // bytes between ring stages (a multiple of 128)
  int64_t tiles;         // ceil(pieces / tile_pieces)
};

constexpr int kFc2Threads = 256;
constexpr int kFc2MaxStages = 16;
constexpr int kFc2RingOffset = kFc2MaxStages * 8;  // barriers first, then the ring (128 B)
// A ring stage is refilled once the store issued this many tiles later has been issued: the
// store of the stage's tile may still be in flight that long.
constexpr int kFc2StoreLag = 2;

// First byte of the source of output piece `piece`.
__device__ __forceinline__ const unsigned char* fc2_source(const Fc2Params& p, int64_t piece) {
  const int64_t per_rank = p.S * p.P * p.D;  // pieces per output rank
  const int64_t r = piece / per_rank;
  const int64_t rem = piece - r * per_rank;
  const int64_t i = rem / p.D;
  const int m = static_cast<int>(rem - i * p.D);
  const int64_t g = r / p.D, j = r - g * p.D;
  const int64_t k = i / p.S, tl = i - k * p.S;
  const int64_t src_rank = g * p.D + m;
  const int64_t src_token = (j + k * p.D) * p.S + tl;
  return p.x + (src_rank * p.N + src_token) * (static_cast<int64_t>(p.piece_vecs) * 16);
}

__global__ void __launch_bounds__(kFc2Threads) k_fc2_reorganize(const Fc2Params p) {
  pdl_launch_dependents();
  pdl_wait_prerequisites();
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kFc2Threads / 32);
  for (int64_t piece = static_cast<int64_t>(blockIdx.x) * (kFc2Threads / 32) + (threadIdx.x >> 5);
       piece < p.pieces; piece += warps) {
    const uint4* src = reinterpret_cast<const uint4*>(fc2_source(p, piece));
    uint4* dst = reinterpret_cast<uint4*>(p.y) + piece * p.piece_vecs;
    // 128 vectors (2 KB) per pass: every lane issues all of its (up to four) loads before its
    // first store, so each warp keeps up to 2 KB in flight.
    for (int base = 0; base < p.piece_vecs; base += 128) {
      uint4 buf[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = base + lane + 32 * u;
        if (v < p.piece_vecs) buf[u] = ldg_stream(src + v);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = base + lane + 32 * u;
        if (v < p.piece_vecs) stg_stream(dst + v, buf[u]);
      }
    }
  }
}

__global__ void __launch_bounds__(32) k_fc2_bulk(const Fc2Params p) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  const uint32_t ring = smem_addr(smem + kFc2RingOffset);
  const int lane = threadIdx.x;
  const int64_t my_tiles =
      blockIdx.x < p.tiles ? (p.tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  auto tile_first = [&](int64_t it) {
    return (static_cast<int64_t>(blockIdx.x) + it * gridDim.x) * p.tile_pieces;
  };
  auto tile_count = [&](int64_t first) {
    const int64_t left = p.pieces - first;
    return static_cast<int>(left < p.tile_pieces ? left : p.tile_pieces);
  };

  if (lane == 0) {
    for (int s = 0; s < p.stages; ++s) mbar_init(smem_addr(full + s), 1);
    fence_mbar_init();
  }
  // While the previous kernel of the stream may still be running, pull the first ring of tiles'
  // sources into L2.
  for (int64_t it = 0; it < my_tiles && it < p.stages; ++it) {
    const int64_t first = tile_first(it);
    const int cnt = tile_count(first);
    for (int q = lane; q < cnt; q += 32) bulk_prefetch_l2(fc2_source(p, first + q), p.piece_bytes);
  }
  __syncwarp();
  pdl_launch_dependents();
  pdl_wait_prerequisites();

  const uint64_t policy = l2_evict_first_policy();
  auto issue = [&](int64_t it) {
    const int64_t first = tile_first(it);
    const int cnt = tile_count(first);
    const int s = static_cast<int>(it % p.stages);
    const uint32_t bar = smem_addr(full + s);
    if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(cnt) * p.piece_bytes);
    __syncwarp();
    const uint32_t dst = ring + static_cast<uint32_t>(s) * p.stage_bytes;
    for (int q = lane; q < cnt; q += 32)
      bulk_g2s(dst + static_cast<uint32_t>(q) * p.piece_bytes, fc2_source(p, first + q),
               p.piece_bytes, bar, policy);
  };

  int64_t issued = 0;
  for (; issued < my_tiles && issued < p.stages; ++issued) issue(issued);
  int64_t it = 0;
  for (; it < my_tiles; ++it) {
    const int s = static_cast<int>(it % p.stages);
    int landed = 0;
    if (lane == 0)
      landed = mbar_wait_bounded(smem_addr(full + s),
                                 static_cast<uint32_t>((it / p.stages) & 1), nullptr);
    landed = __shfl_sync(0xffffffffu, landed, 0);
    if (!landed) {
      if (lane == 0) atomicOr(&g_error_flags, kErrWaitTimeout);
      break;
    }
    if (lane == 0) {
      const int64_t first = tile_first(it);
      fence_proxy_async_smem();
      bulk_s2g(p.y + first * p.piece_bytes, ring + static_cast<uint32_t>(s) * p.stage_bytes,
               static_cast<uint32_t>(tile_count(first)) * p.piece_bytes);
      bulk_commit();
      bulk_wait_read<kFc2StoreLag>();
    }
    __syncwarp();
    if (it >= kFc2StoreLag && issued < my_tiles) issue(issued++);
  }
  if (it < my_tiles && lane == 0) {
    // A wait ran out: let every load still in flight land before the CTA exits (the last issued
    // phase of each stage).
    const int64_t used = issued < p.stages ? issued : p.stages;
    for (int64_t s = 0; s < used; ++s) {
      const int64_t last = issued - 1 - ((issued - 1 - s) % p.stages);
      mbar_wait_bounded(smem_addr(full + s), static_cast<uint32_t>((last / p.stages) & 1),
                        nullptr);
    }
  }
  if (lane == 0) bulk_wait_all();
}

}  // namespace spk
