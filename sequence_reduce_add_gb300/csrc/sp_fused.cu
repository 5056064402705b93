// sp_fused.cu — the C boundary (include/sp_fused.h): argument checks, launch selection and
// kernel launches for the fused reduce + add + RMSNorm + quant stage on sm_103a.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "sp_fc2.cuh"
#include "sp_fused.h"
#include "sp_kernels.cuh"

namespace {

constexpr int64_t kMaxHidden = 8 * 4 * spk::kMaxConsumerThreads;  // VEC 4 x 512 threads: 16384
// Largest byte size of any one buffer (tp * T_pad * H * 2 for the partials): keeps every size
// and address computation of the checks and kernels inside int64.
constexpr int64_t kMaxBufferBytes = int64_t{1} << 62;

// ------------------------------------------------------------------------------ checks
int64_t out_bytes_of(int64_t T_pad, int64_t H, int mode) {
  switch (mode) {
    case SP_QUANT_NONE: return T_pad * H * 2;
    case SP_QUANT_FP8_STATIC:
    case SP_QUANT_FP8_PER_TOKEN: return T_pad * H;
    case SP_QUANT_NVFP4: return T_pad * (H / 2);
    default: return -1;
  }
}

int64_t swizzled_scale_rows(int64_t T_pad) { return (T_pad + 127) / 128 * 128; }
int64_t swizzled_scale_cols(int64_t H) { return (H / 16 + 3) / 4 * 4; }

int64_t scale_bytes_of(int64_t T_pad, int64_t H, int mode, int layout = SP_SCALES_ROW_MAJOR) {
  if (layout != SP_SCALES_ROW_MAJOR && layout != SP_SCALES_SWIZZLED_128X4) return -1;
  if (layout == SP_SCALES_SWIZZLED_128X4 && mode != SP_QUANT_NVFP4) return -1;
  switch (mode) {
    case SP_QUANT_NONE:
    case SP_QUANT_FP8_STATIC: return 0;
    case SP_QUANT_FP8_PER_TOKEN: return T_pad * 4;
    case SP_QUANT_NVFP4:
      return layout == SP_SCALES_SWIZZLED_128X4 ? swizzled_scale_rows(T_pad) * swizzled_scale_cols(H)
                                                : T_pad * (H / 16);
    default: return -1;
  }
}

bool overlaps(const void* p, int64_t pn, const void* q, int64_t qn) {
  if (!p || !q || pn <= 0 || qn <= 0) return false;
  const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
  return a < b + static_cast<uintptr_t>(qn) && b < a + static_cast<uintptr_t>(pn);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// What sp_fused_reduce_norm_ex adds to the plain call (the defaults give the plain call).
struct Extras {
  float partial_scale = 1.0f;
  const void* addend = nullptr;
  int scale_layout = SP_SCALES_ROW_MAJOR;
  int schedule = SP_SCHEDULE_AUTO;
  void* row_counter = nullptr;      // the caller's own [next claim, CTAs done] pair, or null
  uint32_t* status = nullptr;       // the caller's per-call error word, or null
  uint64_t wait_limit_ns = spk::kWaitLimitNs;
  int64_t withhold = -1;            // self-test: CTA 0 withholds this ring fill (else -1)
};

// The checks of sp_fused_reduce_norm, in the documented order. The shape rules restate the
// shard checks of the PR #18671 notes (§5.2): the padded token count is a whole number of
// equal shards, and the valid tokens fit in it.
sp_status check(const void* partials, int tp, int64_t T_pad, int64_t T_valid, int64_t H,
                const void* residual, const void* weight, const void* bias, float eps, int mode,
                const float* scale, const void* out, const void* out_scales,
                const void* residual_out, const Extras& x = Extras()) {
  if (mode == SP_QUANT_FP8_DYNAMIC_PER_TENSOR) return SP_ERR_UNSUPPORTED;
  if (mode < SP_QUANT_NONE || mode > SP_QUANT_NVFP4) return SP_ERR_INVALID_ARG;
  if (tp < 1 || T_pad < 0 || T_valid < 0 || T_valid > T_pad) return SP_ERR_INVALID_ARG;
  if (T_pad % tp != 0) return SP_ERR_INVALID_ARG;
  if (H <= 0 || H % 8 != 0) return SP_ERR_INVALID_ARG;
  if (mode == SP_QUANT_NVFP4 && H % 16 != 0) return SP_ERR_INVALID_ARG;
  if (T_pad > kMaxBufferBytes / (2 * H) / tp) return SP_ERR_INVALID_ARG;  // partials' bytes
  if (!(eps > 0.0f) || !std::isfinite(eps)) return SP_ERR_INVALID_ARG;
  if (!std::isfinite(x.partial_scale)) return SP_ERR_INVALID_ARG;
  if (x.scale_layout != SP_SCALES_ROW_MAJOR && x.scale_layout != SP_SCALES_SWIZZLED_128X4)
    return SP_ERR_UNSUPPORTED;
  if (x.scale_layout == SP_SCALES_SWIZZLED_128X4 && mode != SP_QUANT_NVFP4) return SP_ERR_INVALID_ARG;
  if (x.schedule < SP_SCHEDULE_AUTO || x.schedule > SP_SCHEDULE_DYNAMIC) return SP_ERR_UNSUPPORTED;
  if (T_pad == 0) return SP_OK;
  if (!partials || !weight || !out || !residual_out) return SP_ERR_INVALID_ARG;
  if ((mode == SP_QUANT_FP8_STATIC || mode == SP_QUANT_NVFP4) && !scale) return SP_ERR_INVALID_ARG;
  if ((mode == SP_QUANT_FP8_PER_TOKEN || mode == SP_QUANT_NVFP4) && !out_scales)
    return SP_ERR_INVALID_ARG;
  const int64_t rows = T_pad * H * 2;
  const void* inputs[] = {partials, residual, weight, bias, scale, x.addend};
  const int64_t in_n[] = {rows * tp, rows, H * 2, H * 2, 4, rows};
  // everything the kernel writes: the outputs, the caller's row counter and status word
  const void* outputs[] = {out, out_scales, residual_out, x.row_counter, x.status};
  const int64_t out_n[] = {out_bytes_of(T_pad, H, mode),
                           scale_bytes_of(T_pad, H, mode, x.scale_layout), rows, 8, 4};
  for (int o = 0; o < 5; ++o) {
    for (int i = 0; i < 6; ++i) {
      if (o == 2 && i == 1 && residual_out == residual) continue;  // in-place residual update
      if (overlaps(outputs[o], out_n[o], inputs[i], in_n[i])) return SP_ERR_INVALID_ARG;
    }
    for (int q = o + 1; q < 5; ++q)
      if (overlaps(outputs[o], out_n[o], outputs[q], out_n[q])) return SP_ERR_INVALID_ARG;
  }
  const void* all[] = {partials, residual,     weight,   bias,          scale,   out,
                       out_scales, residual_out, x.addend, x.row_counter, x.status};
  for (const void* ptr : all)
    if (ptr && !aligned16(ptr)) return SP_ERR_ALIGNMENT;
  if (H > kMaxHidden) return SP_ERR_UNSUPPORTED;
  return SP_OK;
}

// ------------------------------------------------------------------------------ devices
constexpr int kMaxDevices = 64;
// GB300's SM count, for launch choices made without querying a device.
constexpr int64_t kSmsHint = 152;
constexpr int kSmemPerSm = 233472;   // 228 KiB of shared memory per SM
constexpr int kSmemPerCtaMax = 232448;  // 227 KiB opt-in limit per CTA
// FlashComm2 reorganisation: bulk-copy tiles of at most this many bytes, ring stages per CTA,
// CTAs per SM. Pieces larger than a tile go through the register kernel.
constexpr int kFc2TileBytes = 24576;
constexpr int kFc2Stages = 3;
constexpr int kFc2CtasPerSm = 3;
constexpr int kSmemReservedPerCta = 1024;

struct DeviceInfo {
  int id = 0;
  std::atomic<int> sms{0};
  std::atomic<bool> staged_attr_set[3][4][2] = {};
  std::atomic<bool> fc2_attr_set{false};
  std::atomic<bool> slice_attr_set[4][3] = {};  // [quant mode][split 2, 4, 8]
  // Row counter slots of the dynamic schedule: slot i belongs to the stream with id slot_stream[i];
  // `counters` is the device address of the table (spk::g_row_counters) in this device's context.
  unsigned int* counters = nullptr;
  unsigned int* error_word = nullptr;  // device address of spk::g_error_flags
  std::mutex slot_mutex;
  unsigned long long slot_stream[spk::kRowCounterSlots] = {};
  int slots_used = 0;
  // Reclaiming slots once all are taken: launches issued on each slot (the device writes the
  // sequence number of each finished one into spk::g_row_counter_done, at `slot_done`), calls
  // holding a slot between choosing it and launching, the last use of each slot (for taking the
  // least recently used), and the library's own stream and buffer for reading the table back.
  unsigned long long* slot_done = nullptr;
  unsigned long long slot_issued[spk::kRowCounterSlots] = {};
  int slot_pending[spk::kRowCounterSlots] = {};
  unsigned long long slot_tick[spk::kRowCounterSlots] = {};
  unsigned long long tick = 0;
  cudaStream_t reclaim_stream = nullptr;
  unsigned long long done_read[spk::kRowCounterSlots] = {};
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_devices_mutex;

sp_status device_info(DeviceInfo** info) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SP_ERR_CUDA;
  DeviceInfo& d = g_devices[dev];
  if (d.sms.load(std::memory_order_acquire) == 0) {  // first call on this device
    std::lock_guard<std::mutex> lock(g_devices_mutex);
    if (d.sms.load(std::memory_order_relaxed) == 0) {
      int sms = 0;
      if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return SP_ERR_CUDA;
      void* counters = nullptr;
      if (cudaGetSymbolAddress(&counters, spk::g_row_counters) != cudaSuccess) return SP_ERR_CUDA;
      d.counters = static_cast<unsigned int*>(counters);
      void* slot_done = nullptr;
      if (cudaGetSymbolAddress(&slot_done, spk::g_row_counter_done) != cudaSuccess)
        return SP_ERR_CUDA;
      d.slot_done = static_cast<unsigned long long*>(slot_done);
      void* error_word = nullptr;
      if (cudaGetSymbolAddress(&error_word, spk::g_error_flags) != cudaSuccess) return SP_ERR_CUDA;
      d.error_word = static_cast<unsigned int*>(error_word);
      d.id = dev;
      d.sms.store(sms, std::memory_order_release);
    }
  }
  *info = &d;
  return SP_OK;
}

int vec_index(int vec) { return vec == 1 ? 0 : vec == 2 ? 1 : 2; }

// The dynamic schedule pays off once every CTA has this many rows (measured on GB300: 1-13 %
// faster from about 11 rows per CTA, 1.5 % slower at 7) and each row moves enough bytes that the
// claims on the one counter stay rare: with (tp + 3) * 2H bytes per row (partials, residual,
// residual_out, bf16 out) below ~24 KB it lost (tp=4, H=1024, 14 KB: 29 % slower, 4.5 vs 6.3
// TB/s at T = 32768; tp=2, H=2048, 20 KB: 1.7 % slower); from 28 KB up it won.
constexpr int64_t kDynamicMinRowsPerCta = 10;
constexpr int64_t kDynamicMinHidden = 2048;
constexpr int64_t kDynamicMinRowBytes = 24 * 1024;

// The least recently used idle slot, or -1. Called with the slot mutex held, once every slot is
// taken. A slot is idle when no call holds it and every launch issued on it has reset it (the
// table the launches write is read back on the library's own non-blocking stream, which waits
// for no other work; this costs a few microseconds and happens only when a new stream finds the
// table full). The slot's counters are then zero, and launches still finishing their last rows
// no longer touch them.
int reclaim_slot(DeviceInfo* dev) {
  // This thread's capture mode is relaxed for the read, so that a CUDA graph being recorded by
  // another thread in global mode neither refuses these calls nor is invalidated by them (the
  // calling stream itself is not being captured: counter_slot checked).
  cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
  if (cudaThreadExchangeStreamCaptureMode(&mode) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  bool read = true;
  if (dev->reclaim_stream == nullptr &&
      cudaStreamCreateWithFlags(&dev->reclaim_stream, cudaStreamNonBlocking) != cudaSuccess) {
    dev->reclaim_stream = nullptr;
    read = false;
  }
  read = read &&
         cudaMemcpyAsync(dev->done_read, dev->slot_done, sizeof(dev->done_read),
                         cudaMemcpyDeviceToHost, dev->reclaim_stream) == cudaSuccess &&
         cudaStreamSynchronize(dev->reclaim_stream) == cudaSuccess;
  if (!read) cudaGetLastError();
  cudaThreadExchangeStreamCaptureMode(&mode);  // back to the thread's own mode
  if (!read) return -1;
  int best = -1;
  for (int i = 0; i < dev->slots_used; ++i)
    if (dev->slot_pending[i] == 0 && dev->done_read[i] == dev->slot_issued[i] &&
        (best < 0 || dev->slot_tick[i] < dev->slot_tick[best]))
      best = i;
  return best;
}

// Row counter slot of `stream` on this device, or -1: the call then uses the static schedule.
// No slot while the stream is being captured (a replay of the graph may run beside later calls
// on the same stream), nor when every slot is taken and none is idle. `*seq` receives the
// launch's sequence number on the slot; the call hands the slot back with release_slot.
int counter_slot(DeviceInfo* dev, cudaStream_t stream, unsigned long long* seq) {
  cudaStreamCaptureStatus capture = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &capture) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  if (capture != cudaStreamCaptureStatusNone) return -1;
  unsigned long long id = 0;
  if (cudaStreamGetId(stream, &id) != cudaSuccess) {
    cudaGetLastError();
    return -1;
  }
  std::lock_guard<std::mutex> lock(dev->slot_mutex);
  int slot = -1;
  for (int i = 0; i < dev->slots_used && slot < 0; ++i)
    if (dev->slot_stream[i] == id) slot = i;
  if (slot < 0) slot = dev->slots_used < spk::kRowCounterSlots ? dev->slots_used++
                                                                 : reclaim_slot(dev);
  if (slot < 0) return -1;
  dev->slot_stream[slot] = id;
  dev->slot_tick[slot] = ++dev->tick;
  ++dev->slot_pending[slot];
  *seq = ++dev->slot_issued[slot];
  return slot;
}

// Hands back a slot that counter_slot gave. A launch that was not issued takes its sequence
// number back if no later call took one (else the slot stays busy until a later launch on it
// has finished).
void release_slot(DeviceInfo* dev, int slot, unsigned long long seq, bool launched) {
  std::lock_guard<std::mutex> lock(dev->slot_mutex);
  if (!launched && dev->slot_issued[slot] == seq) --dev->slot_issued[slot];
  --dev->slot_pending[slot];
}

int consumer_threads(int64_t H, int vec) {
  const int64_t nvec = H / 8;
  const int64_t per = (nvec + vec - 1) / vec;
  return static_cast<int>((per + 31) / 32 * 32);
}

// Split rows: 16-byte vectors of a row per CTA of the cluster (even, so that an NVFP4 block's two
// vectors stay in one CTA), and the consumer threads that cover them.
int split_chunk(int64_t H, int split) {
  const int64_t nvec = H / 8;
  const int64_t chunk = (nvec + split - 1) / split;
  return static_cast<int>((chunk + 1) / 2 * 2);
}
int split_threads(int64_t H, int split, int vec) {
  const int64_t per = (split_chunk(H, split) + vec - 1) / vec;
  return static_cast<int>((per + 31) / 32 * 32);
}
int split_of(const sp_launch_config& cfg) { return cfg.split > 1 ? cfg.split : 1; }

// Dynamic shared memory of the staged kernel: [full barriers][empty barriers][reduction slots]
// [abort flag, pad] [row index per stage] | weight copy [H] bf16, bias copy [H] bf16 |
// ring of `stages` segments.
int wb_offset(int stages) {
  const int head = stages * 16 + 64 * static_cast<int>(sizeof(spk::RedSlot)) + 16 + stages * 8;
  return (head + 127) / 128 * 128;
}

int ring_offset(int stages, int64_t H) {
  return static_cast<int>((wb_offset(stages) + 4 * H + 127) / 128 * 128);
}

int seg_stride(int64_t H) { return static_cast<int>((H * 2 + 127) / 128 * 128); }

int max_stages(int64_t H, int ctas_per_sm) {
  int budget = kSmemPerSm / ctas_per_sm - kSmemReservedPerCta;
  if (budget > kSmemPerCtaMax) budget = kSmemPerCtaMax;
  const int stride = seg_stride(H);
  int s = budget / stride;
  while (s > 0 && ring_offset(s, H) + s * stride > budget) --s;
  return s > 64 ? 64 : s;
}

// Resident CTAs per SM of (kernel, threads, smem) on the current device, cached: the occupancy
// query costs about a microsecond, as much as the launch of a small problem.
struct OccupancyKey {
  const void* kernel;
  int device, threads, smem;
};
constexpr int kOccupancySlots = 256;
OccupancyKey g_occ_keys[kOccupancySlots];
int g_occ_values[kOccupancySlots];
int g_occ_used = 0;
std::mutex g_occ_mutex;

// The calling thread's last lookup, checked before the shared table: a thread that keeps
// launching the same shape takes no lock.
struct LastOccupancy {
  const void* kernel;
  int device, threads, smem, value;
};
thread_local LastOccupancy t_last_occupancy{nullptr, -1, 0, 0, 0};

template <typename Kernel>
cudaError_t resident_ctas(Kernel kernel, int threads, int smem, int device, int* resident) {
  const void* k = reinterpret_cast<const void*>(kernel);
  const LastOccupancy& last = t_last_occupancy;
  if (last.kernel == k && last.device == device && last.threads == threads && last.smem == smem) {
    *resident = last.value;
    return cudaSuccess;
  }
  cudaError_t e = cudaSuccess;
  {
    std::lock_guard<std::mutex> lock(g_occ_mutex);
    for (int i = 0; i < g_occ_used; ++i) {
      const OccupancyKey& c = g_occ_keys[i];
      if (c.kernel == k && c.device == device && c.threads == threads && c.smem == smem) {
        *resident = g_occ_values[i];
        t_last_occupancy = LastOccupancy{k, device, threads, smem, *resident};
        return cudaSuccess;
      }
    }
  }
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(resident, kernel, threads, smem);
  if (e != cudaSuccess) return e;
  t_last_occupancy = LastOccupancy{k, device, threads, smem, *resident};
  std::lock_guard<std::mutex> lock(g_occ_mutex);
  if (g_occ_used < kOccupancySlots) {
    g_occ_keys[g_occ_used] = OccupancyKey{k, device, threads, smem};
    g_occ_values[g_occ_used] = *resident;
    ++g_occ_used;
  }
  return cudaSuccess;
}

// Grid of a persistent launch: SMs x CTAs per SM, where CTAs per SM is the requested number
// capped at what the SM can hold for this kernel (registers, threads, shared memory), so the
// grid is never a ragged second wave; and never more CTAs than rows.
template <typename Kernel>
cudaError_t persistent_grid(Kernel kernel, int threads, int smem, int ctas_per_sm,
                            int64_t rows, const DeviceInfo* dev, int* grid) {
  int resident = 0;
  cudaError_t e = resident_ctas(kernel, threads, smem, dev->id, &resident);
  if (e != cudaSuccess) return e;
  if (resident < 1) return cudaErrorInvalidConfiguration;
  const int per_sm = ctas_per_sm < resident ? ctas_per_sm : resident;
  int64_t g = static_cast<int64_t>(dev->sms.load(std::memory_order_relaxed)) * per_sm;
  if (g > rows) g = rows;
  *grid = static_cast<int>(g);
  return cudaSuccess;
}

// Launch with programmatic stream serialisation: the kernel may be scheduled while the previous
// kernel of the stream finishes; it waits (griddepcontrol.wait) before it reads or writes global
// memory (an L2 prefetch, which changes no memory, may come before).
template <typename Kernel, typename KParams>
cudaError_t launch_pdl(Kernel kernel, int grid, int threads, int smem, cudaStream_t stream,
                       const KParams& p) {
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(static_cast<unsigned>(grid));
  lc.blockDim = dim3(static_cast<unsigned>(threads));
  lc.dynamicSmemBytes = static_cast<size_t>(smem);
  lc.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, kernel, p);
}

template <int kVec, int kMode, bool kDynamic>
cudaError_t set_staged_smem_limit(DeviceInfo* dev) {
  std::atomic<bool>& attr = dev->staged_attr_set[vec_index(kVec)][kMode][kDynamic ? 1 : 0];
  if (attr.load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(spk::k_staged<kVec, kMode, kDynamic>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kSmemPerCtaMax);
  if (e == cudaSuccess) attr.store(true, std::memory_order_release);
  return e;
}

// What the calling thread's last successful launch was (sp_last_launch).
thread_local sp_launch_info t_last_launch{};

// Split rows: clusters of `split` CTAs (one row each at a time), as many as the SMs hold at the
// requested CTAs per SM, and never more than rows; launched with PDL like the rest.
template <int kVec, int kMode, int kSplit, int kBatch>
cudaError_t launch_split(const sp_launch_config& cfg, const spk::Params& p, cudaStream_t stream,
                         DeviceInfo* dev) {
  auto kernel = spk::k_direct<kVec, kMode, kSplit, kBatch>;
  int resident = 0;
  cudaError_t e = resident_ctas(kernel, p.nthreads, 0, dev->id, &resident);
  if (e != cudaSuccess) return e;
  if (resident < 1) return cudaErrorInvalidConfiguration;
  const int per_sm = cfg.ctas_per_sm < resident ? cfg.ctas_per_sm : resident;
  int64_t clusters = static_cast<int64_t>(dev->sms.load(std::memory_order_relaxed)) * per_sm / kSplit;
  if (clusters > p.rows_total) clusters = p.rows_total;
  if (clusters < 1) clusters = 1;
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(static_cast<unsigned>(clusters * kSplit));
  lc.blockDim = dim3(static_cast<unsigned>(p.nthreads));
  lc.dynamicSmemBytes = 0;
  lc.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kSplit;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 2;
  t_last_launch.grid = static_cast<int>(clusters * kSplit);
  e = cudaLaunchKernelEx(&lc, kernel, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int kVec, int kMode, int kSplit, int kBatch>
cudaError_t launch_direct(const sp_launch_config& cfg, spk::Params& p, cudaStream_t stream,
                          DeviceInfo* dev) {
  if constexpr (kSplit > 1) {
    return launch_split<kVec, kMode, kSplit, kBatch>(cfg, p, stream, dev);
  } else {
    auto kernel = spk::k_direct<kVec, kMode, 1, kBatch>;
    int grid = 0;
    cudaError_t e = persistent_grid(kernel, p.nthreads, 0, cfg.ctas_per_sm, p.T_pad, dev, &grid);
    if (e != cudaSuccess) return e;
    t_last_launch.grid = grid;
    e = launch_pdl(kernel, grid, p.nthreads, 0, stream, p);
    return e != cudaSuccess ? e : cudaGetLastError();
  }
}

// One vector per thread and more than four partials: eight partial rows in flight at a time when
// every CTA the call needs is resident at once (that variant takes about twice the registers, so
// fewer CTAs fit per SM), else four.
template <int kVec, int kMode, int kSplit>
cudaError_t launch_direct_batched(const sp_launch_config& cfg, spk::Params& p,
                                  cudaStream_t stream, DeviceInfo* dev) {
  if constexpr (kVec == 1) {
    if (p.tp > 4) {
      int resident = 0;
      const cudaError_t e =
          resident_ctas(spk::k_direct<kVec, kMode, kSplit, 8>, p.nthreads, 0, dev->id, &resident);
      if (e != cudaSuccess) return e;
      const int per_sm = cfg.ctas_per_sm < resident ? cfg.ctas_per_sm : resident;
      const int64_t slots = static_cast<int64_t>(dev->sms.load(std::memory_order_relaxed)) * per_sm;
      if (p.rows_total * kSplit <= slots)
        return launch_direct<kVec, kMode, kSplit, 8>(cfg, p, stream, dev);
    }
  }
  return launch_direct<kVec, kMode, kSplit, 4>(cfg, p, stream, dev);
}

// Split rows through shared memory (k_slice): one cluster of `split` CTAs per row, every row at
// once (grid = rows x split); each CTA holds its slice of the row's segments in shared memory.
int slice_segments(const spk::Params& p) {
  return p.tp + (p.residual ? 1 : 0) + (p.addend ? 1 : 0);
}
int slice_smem_bytes(const spk::Params& p) { return slice_segments(p) * p.split_chunk * 16; }
// Dynamic shared memory k_slice may take: the per-CTA limit less room for its static arrays.
constexpr int kSliceSmemMax = kSmemPerCtaMax - 4096;

template <int kMode, int kSplit>
cudaError_t launch_slice(const spk::Params& p, cudaStream_t stream, DeviceInfo* dev) {
  auto kernel = spk::k_slice<kMode, kSplit>;
  const int smem = slice_smem_bytes(p);
  cudaError_t e = cudaSuccess;
  std::atomic<bool>& attr_set =
      dev->slice_attr_set[kMode][kSplit == 2 ? 0 : (kSplit == 4 ? 1 : 2)];
  if (!attr_set.load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSliceSmemMax);
    if (e != cudaSuccess) return e;
    attr_set.store(true, std::memory_order_release);
  }
  cudaLaunchConfig_t lc{};
  lc.gridDim = dim3(static_cast<unsigned>(p.rows_total * kSplit));
  lc.blockDim = dim3(static_cast<unsigned>(p.nthreads));
  lc.dynamicSmemBytes = static_cast<size_t>(smem);
  lc.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kSplit;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 2;
  t_last_launch.grid = static_cast<int>(p.rows_total * kSplit);
  e = cudaLaunchKernelEx(&lc, kernel, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int kVec, int kMode>
cudaError_t launch_one(const sp_launch_config& cfg, spk::Params& p, int smem, const Extras& x,
                       cudaStream_t stream, DeviceInfo* dev) {
  if constexpr (kVec == 1) {
    if (cfg.kernel == SP_KERNEL_STAGED && x.withhold < 0) {
      switch (split_of(cfg)) {
        case 2: return launch_slice<kMode, 2>(p, stream, dev);
        case 4: return launch_slice<kMode, 4>(p, stream, dev);
        case 8: return launch_slice<kMode, 8>(p, stream, dev);
        default: break;
      }
    }
  }
  int grid = 0;
  const int schedule = x.schedule;
  if (cfg.kernel == SP_KERNEL_DIRECT) {
    if constexpr (kVec <= 2) {
      switch (split_of(cfg)) {
        case 2: return launch_direct_batched<kVec, kMode, 2>(cfg, p, stream, dev);
        case 4: return launch_direct_batched<kVec, kMode, 4>(cfg, p, stream, dev);
        case 8: return launch_direct_batched<kVec, kMode, 8>(cfg, p, stream, dev);
        default: break;
      }
    }
    return launch_direct_batched<kVec, kMode, 1>(cfg, p, stream, dev);
  }
  const int threads = p.nthreads + spk::kProducerThreads;
  cudaError_t e = set_staged_smem_limit<kVec, kMode, false>(dev);
  if (e != cudaSuccess) return e;
  e = persistent_grid(spk::k_staged<kVec, kMode, false>, threads, smem, cfg.ctas_per_sm, p.T_pad,
                      dev, &grid);
  if (e != cudaSuccess) return e;
  unsigned int* counter = nullptr;
  int slot = -1;  // this call's slot of the library's row counter table, if it took one
  unsigned long long seq = 0;
  const bool want_dynamic =
      schedule == SP_SCHEDULE_DYNAMIC ||
      (schedule == SP_SCHEDULE_AUTO && p.rows_total >= kDynamicMinRowsPerCta * grid &&
       p.H >= kDynamicMinHidden &&
       static_cast<int64_t>(p.tp + 3) * 2 * p.H >= kDynamicMinRowBytes);
  if (want_dynamic && p.rows_total + grid < (int64_t{1} << 31)) {
    // The caller's own counter, if given (its calls are ordered by the caller, even inside a
    // captured graph); else this stream's slot of the library's table, if it has one.
    if (x.row_counter) {
      counter = static_cast<unsigned int*>(x.row_counter);
    } else {
      slot = counter_slot(dev, stream, &seq);
      if (slot >= 0) {
        counter = dev->counters + 2 * slot;
        p.slot_done = dev->slot_done + slot;
        p.slot_seq = seq;
      }
    }
  }
  if (counter) {
    // The dynamic variant's own occupancy sizes its grid: every CTA must be resident from the
    // start, since each one begins with a fixed row.
    e = set_staged_smem_limit<kVec, kMode, true>(dev);
    if (e == cudaSuccess)
      e = persistent_grid(spk::k_staged<kVec, kMode, true>, threads, smem, cfg.ctas_per_sm,
                          p.T_pad, dev, &grid);
    p.row_counter = counter;
  }
  void (*kernel)(spk::Params) =
      counter ? spk::k_staged<kVec, kMode, true> : spk::k_staged<kVec, kMode, false>;
  if constexpr (kVec == 2) {
    // the self-test's instantiation (two vectors per thread only)
    if (e == cudaSuccess && x.withhold >= 0) {
      kernel = counter ? spk::k_staged<kVec, kMode, true, true>
                       : spk::k_staged<kVec, kMode, false, true>;
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmemPerCtaMax);
    }
  }
  // From here on a slot taken above is handed back on every path.
  const bool ready = e == cudaSuccess;
  if (ready) e = launch_pdl(kernel, grid, threads, smem, stream, p);
  if (slot >= 0) release_slot(dev, slot, seq, ready && e == cudaSuccess);
  if (!ready) return e;
  t_last_launch.grid = grid;
  t_last_launch.schedule = counter ? SP_SCHEDULE_DYNAMIC : SP_SCHEDULE_STATIC;
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int kVec>
cudaError_t launch_mode(int mode, const sp_launch_config& cfg, spk::Params& p, int smem,
                        const Extras& x, cudaStream_t stream, DeviceInfo* dev) {
  switch (mode) {
    case SP_QUANT_NONE: return launch_one<kVec, spk::kModeNone>(cfg, p, smem, x, stream, dev);
    case SP_QUANT_FP8_STATIC:
      return launch_one<kVec, spk::kModeFp8Static>(cfg, p, smem, x, stream, dev);
    case SP_QUANT_FP8_PER_TOKEN:
      return launch_one<kVec, spk::kModeFp8PerToken>(cfg, p, smem, x, stream, dev);
    default: return launch_one<kVec, spk::kModeNvfp4>(cfg, p, smem, x, stream, dev);
  }
}

sp_status config_is_valid(const sp_launch_config& cfg, int64_t H) {
  if (cfg.kernel != SP_KERNEL_STAGED && cfg.kernel != SP_KERNEL_DIRECT) return SP_ERR_INVALID_ARG;
  if (cfg.vec_per_thread != 1 && cfg.vec_per_thread != 2 && cfg.vec_per_thread != 4)
    return SP_ERR_INVALID_ARG;
  if (cfg.ctas_per_sm < 1 || cfg.ctas_per_sm > 32) return SP_ERR_INVALID_ARG;
  if (cfg.split != 0 && cfg.split != 1 && cfg.split != 2 && cfg.split != 4 && cfg.split != 8)
    return SP_ERR_INVALID_ARG;
  const int split = split_of(cfg);
  if (split > 1 && (cfg.vec_per_thread > 2 ||
                    (cfg.kernel == SP_KERNEL_STAGED && cfg.vec_per_thread != 1)))
    return SP_ERR_UNSUPPORTED;
  const int threads = split > 1 ? split_threads(H, split, cfg.vec_per_thread)
                                : consumer_threads(H, cfg.vec_per_thread);
  if (threads > spk::kMaxConsumerThreads) return SP_ERR_UNSUPPORTED;
  if (cfg.kernel == SP_KERNEL_STAGED && split <= 1) {
    const int most = max_stages(H, cfg.ctas_per_sm);
    if (cfg.stages < 0 || cfg.stages > most || most < 2 || cfg.stages == 1)
      return SP_ERR_UNSUPPORTED;
  }
  return SP_OK;
}

// Launch after the checks have passed.
sp_status run_checked(const sp_launch_config& cfg_in, const void* partials, int tp, int64_t T_pad,
                      int64_t T_valid, int64_t H, const void* residual, const void* weight,
                      const void* bias, float eps, int mode, const float* scale, void* out,
                      void* out_scales, void* residual_out, cudaStream_t stream,
                      const Extras& x) {
  sp_status st = config_is_valid(cfg_in, H);
  if (st != SP_OK) return st;
  if (T_pad == 0) return SP_OK;
  DeviceInfo* dev = nullptr;
  st = device_info(&dev);
  if (st != SP_OK) return st;

  sp_launch_config cfg = cfg_in;
  spk::Params p{};
  p.partials = static_cast<const uint16_t*>(partials);
  p.residual = static_cast<const uint16_t*>(residual);
  p.addend = static_cast<const uint16_t*>(x.addend);
  p.partial_scale = x.partial_scale;
  p.scale_swizzled = x.scale_layout == SP_SCALES_SWIZZLED_128X4 ? 1 : 0;
  p.sf_cols = static_cast<int>(swizzled_scale_cols(H));
  p.rows_total = p.scale_swizzled ? swizzled_scale_rows(T_pad) : T_pad;
  p.weight = static_cast<const uint16_t*>(weight);
  p.bias = static_cast<const uint16_t*>(bias);
  p.scale = scale;
  p.out = out;
  p.out_scales = out_scales;
  p.residual_out = static_cast<uint16_t*>(residual_out);
  p.T_pad = T_pad;
  p.T_valid = T_valid;
  p.plane = T_pad * H;
  p.H = static_cast<int>(H);
  p.nvec = static_cast<int>(H / 8);
  p.tp = tp;
  p.nthreads = consumer_threads(H, cfg.vec_per_thread);
  if (split_of(cfg) > 1) {
    p.split_chunk = split_chunk(H, split_of(cfg));
    p.nthreads = split_threads(H, split_of(cfg), cfg.vec_per_thread);
  }
  p.eps = eps;
  p.error_word = x.status ? x.status : dev->error_word;
  p.wait_limit_ns = x.wait_limit_ns;
  p.withhold = x.withhold;
  int smem = 0;
  if (cfg.kernel == SP_KERNEL_STAGED && split_of(cfg) > 1 &&
      slice_smem_bytes(p) > kSliceSmemMax)  // its row slices do not fit one CTA
    return SP_ERR_UNSUPPORTED;
  if (cfg.kernel == SP_KERNEL_STAGED && split_of(cfg) <= 1) {
    if (cfg.stages == 0) cfg.stages = max_stages(H, cfg.ctas_per_sm);
    p.stages = cfg.stages;
    p.seg_stride = seg_stride(H);
    p.wb_offset = wb_offset(cfg.stages);
    p.ring_offset = ring_offset(cfg.stages, H);
    smem = p.ring_offset + p.stages * p.seg_stride;
  }
  cudaError_t e;
  t_last_launch = sp_launch_info{};
  t_last_launch.schedule = SP_SCHEDULE_STATIC;
  switch (cfg.vec_per_thread) {
    case 1: e = launch_mode<1>(mode, cfg, p, smem, x, stream, dev); break;
    case 2: e = launch_mode<2>(mode, cfg, p, smem, x, stream, dev); break;
    default: e = launch_mode<4>(mode, cfg, p, smem, x, stream, dev); break;
  }
  if (e != cudaSuccess) {
    t_last_launch = sp_launch_info{};
    return SP_ERR_CUDA;
  }
  t_last_launch.config = cfg;
  return SP_OK;
}

sp_status run(const sp_launch_config& cfg, const void* partials, int tp, int64_t T_pad,
              int64_t T_valid, int64_t H, const void* residual, const void* weight,
              const void* bias, float eps, int mode, const float* scale, void* out,
              void* out_scales, void* residual_out, cudaStream_t stream,
              const Extras& x = Extras()) {
  const sp_status st = check(partials, tp, T_pad, T_valid, H, residual, weight, bias, eps, mode,
                             scale, out, out_scales, residual_out, x);
  if (st != SP_OK) return st;
  return run_checked(cfg, partials, tp, T_pad, T_valid, H, residual, weight, bias, eps, mode,
                     scale, out, out_scales, residual_out, stream, x);
}

}  // namespace

extern "C" {

sp_status sp_select_launch(int tp, int64_t T_pad, int64_t H, int quant_mode,
                           sp_launch_config* config) {
  if (!config || tp < 1 || H <= 0 || H % 8 != 0 || T_pad < 0 ||
      T_pad > kMaxBufferBytes / (2 * H) / tp)
    return SP_ERR_INVALID_ARG;
  if (quant_mode < SP_QUANT_NONE || quant_mode > SP_QUANT_FP8_DYNAMIC_PER_TENSOR)
    return SP_ERR_INVALID_ARG;
  if (H > kMaxHidden) return SP_ERR_UNSUPPORTED;
  // Staged kernel, two 16-byte vectors per consumer thread (four beyond H = 8192), and about
  // 100-130 KB of ring per SM: CTAs per SM = 16384 / H (one row in flight per CTA; 16 at
  // H = 1024, 4 at 4096, 2 at 8192), 3 row segments per CTA for 1024 < H <= 4096 and 4
  // otherwise (4 rather than 3 at H = 4608-5120 measured 0-11 % faster). This measured best on
  // GB300 from H = 1024 to 16384; the launch caps CTAs per SM at what the SM holds.
  sp_launch_config c{};
  c.kernel = SP_KERNEL_STAGED;
  c.vec_per_thread = 2;
  if (consumer_threads(H, c.vec_per_thread) > spk::kMaxConsumerThreads) c.vec_per_thread = 4;
  c.stages = (H <= 1024 || H > 4096) ? 4 : 3;
  c.ctas_per_sm = static_cast<int>(16384 / H);
  if (c.ctas_per_sm > 32) c.ctas_per_sm = 32;
  if (c.ctas_per_sm < 1) c.ctas_per_sm = 1;
  while (c.ctas_per_sm > 1 && max_stages(H, c.ctas_per_sm) < c.stages) --c.ctas_per_sm;
  if (max_stages(H, c.ctas_per_sm) < c.stages) c.stages = max_stages(H, c.ctas_per_sm);
  if (c.stages < 2) {
    c.kernel = SP_KERNEL_DIRECT;
    c.stages = 0;
  }
  // Calls with few rows (decode-sized batches up to a few hundred tokens) are latency-bound:
  // every CTA does about one row, so the call time is one round trip per batch of loads plus the
  // epilogue. The direct kernel (no ring to set up; loads four or eight partial rows at a time)
  // wins while its loads fit in about one wave; with only a few long rows, splitting each row
  // across a cluster of 2, 4 or 8 CTAs draws on that many more SMs (one SM pulls in about
  // 45 GB/s); past that the staged kernel, with one round of rows given the deepest ring that
  // fits (ceil(T / SMs) CTAs per SM), or the large-call rule below. From GB300 sweeps of tp 2-16,
  // H 1024-16384, T 8-512, bf16 and per-token FP8 output, each launch timed back to back and
  // replayed from a CUDA graph (inputs L2-resident, as the output of the kernel before them
  // would be); against the previous rule this choice is 4.3 % faster summed over the 1186 swept
  // shapes and within 0.8 % of the best measured launch of each:
  //   H <= 4096:        direct while T * H <= 2^20 (tp >= 12 from H = 3072: and tp * T * H <=
  //                     12.6 M), or, except for NVFP4 output, T * H <= 1.4 M at tp <= 4 (1.2 M at
  //                     tp <= 8); two vectors per thread at tp <= 4 and 2^18 <= T * H <= 800 K
  //                     (not for NVFP4; up to 27 % faster than the deep ring this replaced at
  //                     tp <= 5); above H = 3072 (tp >= 2) split rows, 4 CTAs per row up to 16
  //                     rows and, except for NVFP4, up to 24 (32 at tp <= 5), then 8 per row up
  //                     to 48 rows at tp <= 5; else, for H >= 3072 and at most four rounds of 152
  //                     rows, ceil(T / 152) CTAs per SM with every stage that fits (15-40 %
  //                     faster at T = 320-448);
  //   4096 < H <= 8192: split rows: 2 <= tp <= 5, 8 CTAs per row up to 16 rows (NVFP4 below
  //                     H = 6144: 4); 6 <= tp < 12, 8 up to 12 rows and 4 up to 64 (at
  //                     H = 5120, 4 up to 32 and 2 up to 64), and at H <= 5120 4 for 65-96 rows
  //                     (NVFP4 from H = 4609); tp >= 12, 8 up to 16 rows (4 below H = 7168) and
  //                     4 up to 64 (2 for 33-64 rows at H <= 5120, not for NVFP4), 4 for 65-80
  //                     rows at H >= 7168 and for 65-96 at H <= 5120 (NVFP4 from H = 4609, and
  //                     up to 128 rows). Then direct with two vectors per thread up to 128 rows
  //                     (160 at tp <= 3 and H >= 7168; at tp >= 12 up to 96, or 128 below 8192:
  //                     15-36 % faster than the one-CTA-per-SM deep ring it replaced), split 2 up
  //                     to 224 rows at H = 5120, and at H 5121-6144 (tp < 12) split 2 up to 152
  //                     rows (NVFP4: 4) and 4 up to 160; at H >= 7168, 129-144 rows split 4 for
  //                     4 <= tp < 12 (tp <= 5: 2 for 145-152 rows and 4 up to 160); the deep ring
  //                     at one CTA per SM for tp >= 12 and 97-128 rows at H = 8192, then split 4
  //                     for 129-144 rows (up to 160 at H <= 6144); one round of rows for
  //                     H <= 6144 (17-41 % faster at H = 6144, T = 320-384);
  //   H > 8192:         split rows (tp >= 2): 8 CTAs per row up to 16 rows (24 at tp >= 6), 4 up
  //                     to 64 (8 above H = 12288 at tp <= 5), 8 up to 80 at H <= 12288 (16-36 %
  //                     faster) and for 153-160 rows, just past one round of the one-CTA-per-SM
  //                     ring; then at tp <= 5 direct with four vectors per thread up to 96
  //                     rows (128 at H <= 12288); else staged.
  // The split bands were widened once the split kernel combined a row's sums with asynchronous
  // pushes instead of a cluster barrier per row: over 796 shapes swept again (tp 2-16, H 2048-
  // 16384, T 8-128, bf16, per-token FP8 and NVFP4 output) the new bands are 2.1 % faster summed
  // (up to 24 % on one shape: tp 16, H 5120, 96 rows) and slower on none by more than 1 %. A
  // second sweep of 456 shapes around one round of rows (T 112-256, H 4096-16384, tp 2-16, the
  // three output kinds) found the staged ring 25-45 % slower than split rows at 129-144 rows and
  // H >= 7168: the bands for 129-160 rows come from it (4.9 % faster summed, none slower).
  // Staged split rows (k_slice: a cluster per row, the row's slices held in shared memory) then
  // take the calls just past what the direct split kernel covers in one round: 4 CTAs per row at
  // H = 3073-4096 for 145-192 rows at tp >= 12 and, for NVFP4, 161-256 rows at tp 6-11; at
  // H >= 7168 for 145-160 rows at tp 6-11 and 161-192 rows at tp <= 5. And a few decode bands,
  // kept where an A/B against direct rows was faster both back to back and from a CUDA graph:
  // at 4096 < H <= 8192 and tp 2-5, 17-24 rows at H >= 6144 (8 CTAs per row) and 17-32 rows
  // below (4 per row), 6-21 % faster; NVFP4 at tp >= 12 up to 16 rows and H <= 5120 (4 per row),
  // 9-13 % faster. (Some other decode shapes that the sweep favoured ran faster from a graph but
  // 7-43 % slower back to back, and were left out.) Once the direct and slice kernels let the
  // next kernel in only at their end, a sweep of 270 shapes around the direct kernel's upper
  // bound (T 128-512, H 2048-8192) gave two more bands: 4 CTAs per row for 97-128 rows at
  // 4096 < H <= 5120 and tp >= 6 (3-7 % faster on L2-resident inputs, 4-17 % from HBM), and 2
  // per row for NVFP4 output past 128 rows in the direct band at H >= 3072 (1-24 % and up to
  // 38 % faster); the others it suggested were slower on L2-resident inputs and left out. The
  // staged split rows, over 195 swept shapes (tp 2-16, H 4096-16384, T 16-320): 1.5 % faster
  // summed, none slower; against the previous rule 8-38 % faster on L2-resident inputs (tp 8,
  // H 8192, 160 rows: 8.31 -> 5.18 µs); on inputs from HBM 7-37 % faster at H = 4096, -9 to
  // +1 % at tp 8 and H >= 7168, and 4-11 % slower at tp <= 5.
  const int64_t elems = static_cast<int64_t>(tp) * T_pad * H;
  const int64_t rows_x_h = T_pad * H;
  bool direct = false;
  bool ring_1 = false;  // staged at one CTA per SM with the deepest ring
  int one_round = 0;    // staged at this many CTAs per SM with the deepest ring
  int vec = 0;          // direct kernel: vectors per thread (0: by H)
  int split = 0;
  int slice = 0;  // the staged kernel's split-row form (k_slice), this many CTAs per row
  const bool nvfp4 = quant_mode == SP_QUANT_NVFP4;
  if (H <= 4096) {
    direct = (rows_x_h <= (int64_t{1} << 20) && (tp < 12 || H < 3072 || elems <= 12600000)) ||
             (!nvfp4 && tp <= 4 && rows_x_h <= 1400000) ||
             (!nvfp4 && tp <= 8 && rows_x_h <= 1200000) ||
             (H <= 1024 && rows_x_h <= (int64_t{1} << 22));
    if (direct && !nvfp4 && tp <= 4 && rows_x_h >= (int64_t{1} << 18) && rows_x_h <= 800000)
      vec = 2;
    if (direct && H > 3072 && tp >= 2) {
      if (T_pad <= 16 || (!nvfp4 && (T_pad <= 24 || (tp <= 5 && T_pad <= 32))))
        split = 4;
      else if (!nvfp4 && tp <= 5 && T_pad <= 48)
        split = 8;
    }
    if (!direct && H >= 3072 && T_pad <= 4 * kSmsHint)
      one_round = static_cast<int>((T_pad + kSmsHint - 1) / kSmsHint);
    if (H > 3072 && ((tp >= 12 && T_pad > 144 && T_pad <= 192) ||
                     (nvfp4 && tp >= 12 && T_pad <= 16)))
      slice = 4;
    if (slice == 0 && direct && split == 0 && nvfp4 && tp >= 4 && H >= 3072 && T_pad > 128)
      slice = 2;
  } else if (H <= 8192) {
    const bool mid_h = H <= 5120;                     // H 4097-5120
    const bool mid_h_nv = mid_h && (!nvfp4 || H > 4608);  // NVFP4 only from H 4609
    if (tp <= 5) {
      split = (tp >= 2 && T_pad <= 16) ? ((H >= 6144 || !nvfp4) ? 8 : 4) : 0;
    } else if (tp < 12) {
      split = T_pad <= 12 ? 8 : (T_pad <= 64 ? ((H >= 6144 || T_pad <= 32) ? 4 : 2) : 0);
      if (mid_h_nv && T_pad > 64 && T_pad <= 96) split = 4;
    } else {
      split = T_pad <= 16 ? (H >= 7168 ? 8 : 4) : (T_pad <= 64 ? 4 : 0);
      if (mid_h && !nvfp4 && T_pad > 32 && T_pad <= 64) split = 2;
      if (T_pad > 64 && ((mid_h_nv && T_pad <= 96) || (H >= 7168 && T_pad <= 80))) split = 4;
      if (mid_h_nv && nvfp4 && T_pad > 96 && T_pad <= 128) split = 4;
    }
    if (split) {
      direct = true;
    } else if (tp < 12) {
      if (T_pad <= 128 || (tp <= 3 && H >= 7168 && T_pad <= 160)) {
        direct = true;
      } else if (H <= 5120 && T_pad <= 224) {
        direct = true;
        split = 2;
      } else if (H <= 6144 && T_pad <= 160) {
        direct = true;
        split = (T_pad <= 152 && !nvfp4) ? 2 : 4;
      } else if (H >= 7168 && tp >= 4 && T_pad <= (tp <= 5 ? 160 : 144)) {
        direct = true;
        split = (T_pad > 144 && T_pad <= 152) ? 2 : 4;
      }
    } else if (T_pad <= 96 || (T_pad <= 128 && H < 8192)) {
      direct = true;
    } else if (T_pad <= 128) {
      ring_1 = true;
    } else if (T_pad <= 144 || (H <= 6144 && T_pad <= 160)) {
      direct = true;
      split = 4;
    }
    if (!direct && !ring_1 && H <= 6144 && T_pad > kSmsHint && T_pad <= 4 * kSmsHint)
      one_round = static_cast<int>((T_pad + kSmsHint - 1) / kSmsHint);
    if (H >= 7168 && ((tp <= 5 && T_pad > 160 && T_pad <= 192) ||
                      (tp >= 6 && tp < 12 && T_pad > 144 && T_pad <= 160)))
      slice = 4;
    if (tp >= 2 && tp <= 5 && T_pad > 16 && T_pad <= (H >= 6144 ? 24 : 32))
      slice = H >= 6144 ? 8 : 4;
    if (tp >= 6 && T_pad > 96 && T_pad <= 128 && H <= 5120) slice = 4;
    if (nvfp4 && tp >= 12 && T_pad <= 16 && H <= 5120) slice = 4;
  } else {
    split = tp < 2                                ? 0
          : T_pad <= (tp <= 5 ? 16 : 24)           ? 8
          : T_pad <= 64                             ? ((H > 12288 && tp <= 5) ? 8 : 4)
          : (T_pad <= 80 && H <= 12288)             ? 8
          : (H <= 12288 && T_pad > 152 && T_pad <= 160) ? 8
                                                    : 0;
    direct = split > 0 || (tp <= 5 && (T_pad <= 96 || (T_pad <= 128 && H <= 12288)));
  }
  // a row slice of every segment (the partials, the residual and an addend) must fit one CTA
  if (slice && static_cast<int64_t>(tp + 2) * split_chunk(H, slice) * 16 > kSliceSmemMax) slice = 0;
  if (slice) {
    c.kernel = SP_KERNEL_STAGED;
    c.vec_per_thread = 1;
    c.ctas_per_sm = 8;
    c.stages = 0;
    c.split = slice;
  } else if (direct) {
    c.kernel = SP_KERNEL_DIRECT;
    c.vec_per_thread = split > 0 ? 1 : (vec ? vec : (H <= 4096 ? 1 : (H <= 8192 ? 2 : 4)));
    c.ctas_per_sm = (H <= 4096 && split == 0) ? 16 : 8;
    c.stages = 0;
    c.split = split;
  } else if (ring_1 && c.kernel == SP_KERNEL_STAGED && max_stages(H, 1) >= c.stages) {
    c.ctas_per_sm = 1;
    c.stages = 0;  // as many as fit
  } else if (one_round > 0 && c.kernel == SP_KERNEL_STAGED &&
             max_stages(H, one_round) >= c.stages) {
    // All rows fit in one round of this grid: each CTA has at most one row, so use only as many
    // CTAs per SM as the rows need and give each the deepest ring that fits.
    c.ctas_per_sm = one_round;
    c.stages = 0;
  } else if (!direct && c.kernel == SP_KERNEL_STAGED && H >= 4096 &&
             T_pad > kSmsHint * c.ctas_per_sm && T_pad < 2 * kSmsHint * c.ctas_per_sm) {
    // Between one and two rounds of rows: the second round runs part-empty. Take the CTAs per
    // SM (at most the large-call count, at least 2, and no fewer than leave each CTA 3 rows)
    // whose last round is fullest, ties to more CTAs, with the deepest ring that fits. With more
    // rows per CTA the SMs' bandwidth needs several CTAs each (1 CTA/SM at 6.7 rows: 50 % slower);
    // one CTA per SM at 2-3 rows paid only for long rows (H >= 7168, tp >= 8: up to 13 % faster;
    // tp = 4 or H = 6144: -13 % to +4 %).
    auto rounds = [&](int ctas) {
      return static_cast<double>(T_pad) / static_cast<double>(kSmsHint * ctas);
    };
    auto fill = [&](int ctas) { return rounds(ctas) / std::ceil(rounds(ctas)); };
    int best = c.ctas_per_sm;
    const int fewest = (H >= 7168 && tp >= 8) ? 1 : 2;
    for (int ctas = c.ctas_per_sm - 1; ctas >= fewest && rounds(ctas) <= 3.0; --ctas)
      if (fill(ctas) > fill(best) + 1e-9) best = ctas;
    if (best != c.ctas_per_sm && max_stages(H, best) >= c.stages) {
      c.ctas_per_sm = best;
      c.stages = 0;
    }
  }
  *config = c;
  return SP_OK;
}

sp_status sp_fused_reduce_norm(const void* partials, int tp, int64_t T_pad, int64_t T_valid,
                               int64_t H, const void* residual, const void* weight,
                               const void* bias, float eps, int quant_mode, const float* scale,
                               void* out, void* out_scales, void* residual_out,
                               sp_stream_t stream) {
  return sp_fused_reduce_norm_ex(nullptr, partials, tp, T_pad, T_valid, H, residual, weight, bias,
                                 eps, quant_mode, scale, out, out_scales, residual_out, stream);
}

sp_status sp_fused_reduce_norm_with_config(const sp_launch_config* config, const void* partials,
                                           int tp, int64_t T_pad, int64_t T_valid, int64_t H,
                                           const void* residual, const void* weight,
                                           const void* bias, float eps, int quant_mode,
                                           const float* scale, void* out, void* out_scales,
                                           void* residual_out, sp_stream_t stream) {
  if (!config) return SP_ERR_INVALID_ARG;
  return run(*config, partials, tp, T_pad, T_valid, H, residual, weight, bias, eps, quant_mode,
             scale, out, out_scales, residual_out, reinterpret_cast<cudaStream_t>(stream));
}

// Device address of a page-locked host (or device) buffer; false for memory the device cannot
// reach (pageable) or an unknown pointer.
static bool device_view(const void* p, const void** dev_ptr) {
  if (!p) {
    *dev_ptr = nullptr;
    return true;
  }
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) {
    *dev_ptr = p;
    return true;
  }
  if (a.type != cudaMemoryTypeHost || !a.devicePointer) return false;
  // the same offset into the mapping as p has into its allocation
  *dev_ptr = static_cast<const char*>(a.devicePointer) +
             (static_cast<const char*>(p) - static_cast<const char*>(a.hostPointer));
  return true;
}

void sp_options_init(sp_fused_options* options) {
  if (!options) return;
  options->partial_scale = 1.0f;
  options->addend = nullptr;
  options->scale_layout = SP_SCALES_ROW_MAJOR;
  options->host_buffers = 0;
  options->schedule = SP_SCHEDULE_AUTO;
  options->launch = nullptr;
  options->row_counter = nullptr;
  options->status = nullptr;
}

}  // extern "C"

namespace {

Extras extras_of(const sp_fused_options& o) {
  Extras x;
  x.partial_scale = o.partial_scale;
  x.addend = o.addend;
  x.scale_layout = o.scale_layout;
  x.schedule = o.schedule;
  x.row_counter = o.row_counter;
  x.status = o.status;
  return x;
}

// The checks of the options-taking entry points, in order: those of sp_fused_reduce_norm (with
// the options' buffers), then host_buffers, then the forced launch.
sp_status check_ex(const sp_fused_options& o, const Extras& x, const void* partials, int tp,
                   int64_t T_pad, int64_t T_valid, int64_t H, const void* residual,
                   const void* weight, const void* bias, float eps, int quant_mode,
                   const float* scale, const void* out, const void* out_scales,
                   const void* residual_out) {
  sp_status st = check(partials, tp, T_pad, T_valid, H, residual, weight, bias, eps, quant_mode,
                       scale, out, out_scales, residual_out, x);
  if (st != SP_OK) return st;
  if (o.host_buffers != 0 && o.host_buffers != 1) return SP_ERR_UNSUPPORTED;
  if (o.launch) {
    st = config_is_valid(*o.launch, H);
    if (st != SP_OK) return st;
    if (o.host_buffers && o.launch->kernel != SP_KERNEL_DIRECT) return SP_ERR_UNSUPPORTED;
  }
  return SP_OK;
}

// sp_fused_reduce_norm_ex after its checks. staged_only: run the staged kernel whatever
// sp_select_launch picks (the self-test of its abort path).
sp_status run_ex(const sp_fused_options& o, Extras x, bool staged_only, const void* partials,
                 int tp, int64_t T_pad, int64_t T_valid, int64_t H, const void* residual,
                 const void* weight, const void* bias, float eps, int quant_mode,
                 const float* scale, void* out, void* out_scales, void* residual_out,
                 cudaStream_t s) {
  if (T_pad == 0) return SP_OK;
  if (!o.host_buffers) {
    sp_launch_config cfg;
    if (o.launch) {
      cfg = *o.launch;
    } else {
      const sp_status st = sp_select_launch(tp, T_pad, H, quant_mode, &cfg);
      if (st != SP_OK) return st;
    }
    if (staged_only && cfg.kernel != SP_KERNEL_STAGED) {
      if (o.launch) return SP_ERR_UNSUPPORTED;
      cfg = sp_launch_config{};
      cfg.kernel = SP_KERNEL_STAGED;
      cfg.vec_per_thread = 2;
      cfg.ctas_per_sm = 1;
      cfg.stages = 0;
      const sp_status st = config_is_valid(cfg, H);
      if (st != SP_OK) return st;
    }
    // the self-test's kernel is built for two vectors per consumer thread (H <= 8192)
    if (staged_only && cfg.vec_per_thread != 2) return SP_ERR_UNSUPPORTED;
    return run_checked(cfg, partials, tp, T_pad, T_valid, H, residual, weight, bias, eps,
                       quant_mode, scale, out, out_scales, residual_out, s, x);
  }
  if (staged_only) return SP_ERR_UNSUPPORTED;
  // Host buffers: map every pointer to its device address and use plain 128-bit loads (the
  // direct kernel): the host link, not HBM, bounds this call, and a few hundred KB of loads in
  // flight per GPU cover its latency.
  const void* host[10] = {partials,     residual, weight,  bias, scale, out, out_scales,
                          residual_out, x.addend, x.status};
  const void* dev[10];
  for (int i = 0; i < 10; ++i)
    if (!device_view(host[i], &dev[i])) return SP_ERR_INVALID_ARG;
  sp_launch_config cfg{};
  cfg.kernel = SP_KERNEL_DIRECT;
  cfg.vec_per_thread = consumer_threads(H, 2) > spk::kMaxConsumerThreads ? 4 : 2;
  cfg.ctas_per_sm = 4;
  cfg.stages = 0;
  if (o.launch) cfg = *o.launch;
  x.addend = dev[8];
  x.status = static_cast<uint32_t*>(const_cast<void*>(dev[9]));
  return run(cfg, dev[0], tp, T_pad, T_valid, H, dev[1], dev[2], dev[3], eps, quant_mode,
             static_cast<const float*>(dev[4]), const_cast<void*>(dev[5]),
             const_cast<void*>(dev[6]), const_cast<void*>(dev[7]), s, x);
}

}  // namespace

extern "C" {

sp_status sp_fused_reduce_norm_ex(const sp_fused_options* options, const void* partials, int tp,
                                  int64_t T_pad, int64_t T_valid, int64_t H, const void* residual,
                                  const void* weight, const void* bias, float eps, int quant_mode,
                                  const float* scale, void* out, void* out_scales,
                                  void* residual_out, sp_stream_t stream) {
  sp_fused_options o;
  sp_options_init(&o);
  if (options) o = *options;
  const Extras x = extras_of(o);
  const sp_status st = check_ex(o, x, partials, tp, T_pad, T_valid, H, residual, weight, bias,
                                eps, quant_mode, scale, out, out_scales, residual_out);
  if (st != SP_OK) return st;
  return run_ex(o, x, false, partials, tp, T_pad, T_valid, H, residual, weight, bias, eps,
                quant_mode, scale, out, out_scales, residual_out,
                reinterpret_cast<cudaStream_t>(stream));
}

sp_status sp_fused_reduce_norm_host(const void* partials, int tp, int64_t T_pad, int64_t T_valid,
                                    int64_t H, const void* residual, const void* weight,
                                    const void* bias, float eps, int quant_mode,
                                    const float* scale, void* out, void* out_scales,
                                    void* residual_out, sp_stream_t stream) {
  sp_fused_options o;
  sp_options_init(&o);
  o.host_buffers = 1;
  return sp_fused_reduce_norm_ex(&o, partials, tp, T_pad, T_valid, H, residual, weight, bias, eps,
                                 quant_mode, scale, out, out_scales, residual_out, stream);
}

sp_status sp_check_args_ex(const sp_fused_options* options, const void* partials, int tp,
                           int64_t T_pad, int64_t T_valid, int64_t H, const void* residual,
                           const void* weight, const void* bias, float eps, int quant_mode,
                           const float* scale, const void* out, const void* out_scales,
                           const void* residual_out) {
  sp_fused_options o;
  sp_options_init(&o);
  if (options) o = *options;
  return check_ex(o, extras_of(o), partials, tp, T_pad, T_valid, H, residual, weight, bias, eps,
                  quant_mode, scale, out, out_scales, residual_out);
}

sp_status sp_selftest_fused_timeout(uint64_t limit_ns, int64_t withhold,
                                    const sp_fused_options* options, const void* partials, int tp,
                                    int64_t T_pad, int64_t T_valid, int64_t H,
                                    const void* residual, const void* weight, const void* bias,
                                    float eps, int quant_mode, const float* scale, void* out,
                                    void* out_scales, void* residual_out, sp_stream_t stream) {
  if (limit_ns == 0 || limit_ns > spk::kWaitLimitNs || withhold < 0) return SP_ERR_INVALID_ARG;
  sp_fused_options o;
  sp_options_init(&o);
  if (options) o = *options;
  Extras x = extras_of(o);
  const sp_status st = check_ex(o, x, partials, tp, T_pad, T_valid, H, residual, weight, bias,
                                eps, quant_mode, scale, out, out_scales, residual_out);
  if (st != SP_OK) return st;
  x.wait_limit_ns = limit_ns;
  x.withhold = withhold;
  return run_ex(o, x, true, partials, tp, T_pad, T_valid, H, residual, weight, bias, eps,
                quant_mode, scale, out, out_scales, residual_out,
                reinterpret_cast<cudaStream_t>(stream));
}

sp_status sp_last_launch(sp_launch_info* info) {
  if (!info) return SP_ERR_INVALID_ARG;
  *info = t_last_launch;
  return SP_OK;
}

sp_status sp_check_args(const void* partials, int tp, int64_t T_pad, int64_t T_valid, int64_t H,
                        const void* residual, const void* weight, const void* bias, float eps,
                        int quant_mode, const float* scale, const void* out,
                        const void* out_scales, const void* residual_out) {
  return check(partials, tp, T_pad, T_valid, H, residual, weight, bias, eps, quant_mode, scale,
               out, out_scales, residual_out);
}

int64_t sp_pad_tokens(int64_t T, int tp) {
  if (T < 0 || tp < 1) return -1;
  return (T + tp - 1) / tp * tp;
}

sp_status sp_shard_rows(int64_t T_pad, int tp, int rank, int64_t* start, int64_t* len) {
  if (!start || !len || tp < 1 || T_pad < 0 || T_pad % tp != 0 || rank < 0 || rank >= tp)
    return SP_ERR_INVALID_ARG;
  const int64_t s = T_pad / tp;
  *start = static_cast<int64_t>(rank) * s;
  *len = s;
  return SP_OK;
}

int64_t sp_out_bytes(int64_t T_pad, int64_t H, int quant_mode) {
  if (T_pad < 0 || H < 0) return -1;
  return out_bytes_of(T_pad, H, quant_mode);
}

int64_t sp_out_scales_bytes(int64_t T_pad, int64_t H, int quant_mode) {
  if (T_pad < 0 || H < 0) return -1;
  return scale_bytes_of(T_pad, H, quant_mode);
}

// ------------------------------------------------------------------ FlashComm2 reorganisation
sp_status sp_fc2_batch_ids(int global_tp, int otp_size, int* ids) {
  if (!ids || global_tp < 1 || otp_size < 1 || global_tp % otp_size != 0) return SP_ERR_INVALID_ARG;
  const int D = global_tp / otp_size;
  for (int j = 0; j < D; ++j)
    for (int k = 0; k < otp_size; ++k) ids[j * otp_size + k] = j + k * D;
  return SP_OK;
}

sp_status sp_fc2_check_args(const void* x, int global_tp, int otp_size, int64_t N, int64_t H,
                            int elem_bytes, const void* y) {
  if (global_tp < 1 || otp_size < 1 || global_tp % otp_size != 0) return SP_ERR_INVALID_ARG;
  if (N < 0 || N % global_tp != 0 || H <= 0 || H % global_tp != 0) return SP_ERR_INVALID_ARG;
  if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8)
    return SP_ERR_INVALID_ARG;
  if (N > kMaxBufferBytes / H / elem_bytes) return SP_ERR_INVALID_ARG;
  if (N == 0) return SP_OK;
  if (!x || !y) return SP_ERR_INVALID_ARG;
  const int64_t bytes = N * H * elem_bytes;
  if (overlaps(x, bytes, y, bytes)) return SP_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(y) || ((H / global_tp) * elem_bytes) % 16 != 0)
    return SP_ERR_ALIGNMENT;
  return SP_OK;
}

sp_status sp_fc2_reorganize(const void* x, int global_tp, int otp_size, int64_t N, int64_t H,
                            int elem_bytes, void* y, sp_stream_t stream) {
  sp_status st = sp_fc2_check_args(x, global_tp, otp_size, N, H, elem_bytes, y);
  if (st != SP_OK || N == 0) return st;
  DeviceInfo* dev = nullptr;
  st = device_info(&dev);
  if (st != SP_OK) return st;
  spk::Fc2Params p{};
  p.x = static_cast<const unsigned char*>(x);
  p.y = static_cast<unsigned char*>(y);
  p.N = N;
  p.pieces = static_cast<int64_t>(global_tp) * N;
  p.S = N / global_tp;
  p.P = otp_size;
  p.D = global_tp / otp_size;
  p.piece_vecs = static_cast<int>((H / global_tp) * elem_bytes / 16);
  p.piece_bytes = static_cast<uint32_t>(p.piece_vecs) * 16u;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int grid = 0;
  cudaError_t e = cudaSuccess;
  if (p.piece_bytes <= static_cast<uint32_t>(kFc2TileBytes)) {
    // Bulk-copy ring of kFc2Stages tiles of whole pieces, at most kFc2TileBytes each.
    const int max_q = kFc2TileBytes / static_cast<int>(p.piece_bytes);
    p.stages = kFc2Stages;
    p.stage_bytes = (static_cast<uint32_t>(max_q) * p.piece_bytes + 127u) & ~127u;
    const int smem = spk::kFc2RingOffset + p.stages * static_cast<int>(p.stage_bytes);
    if (!dev->fc2_attr_set.load(std::memory_order_acquire)) {
      e = cudaFuncSetAttribute(spk::k_fc2_bulk, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kSmemPerCtaMax);
      if (e == cudaSuccess) dev->fc2_attr_set.store(true, std::memory_order_release);
    }
    if (e == cudaSuccess)
      e = persistent_grid(spk::k_fc2_bulk, 32, smem, kFc2CtasPerSm,
                          (p.pieces + max_q - 1) / max_q, dev, &grid);
    if (e == cudaSuccess) {
      // Every CTA gets the same number of tiles: the fewest rounds of at most max_q pieces
      // that cover all pieces, with the pieces spread evenly over those tiles.
      const int64_t rounds = (p.pieces + static_cast<int64_t>(grid) * max_q - 1) /
                             (static_cast<int64_t>(grid) * max_q);
      p.tile_pieces = static_cast<int>((p.pieces + rounds * grid - 1) / (rounds * grid));
      p.tiles = (p.pieces + p.tile_pieces - 1) / p.tile_pieces;
      e = launch_pdl(spk::k_fc2_bulk, grid, 32, smem, s, p);
    }
  } else {
    e = persistent_grid(spk::k_fc2_reorganize, spk::kFc2Threads, 0, 8,
                        (p.pieces + spk::kFc2Threads / 32 - 1) / (spk::kFc2Threads / 32), dev,
                        &grid);
    if (e == cudaSuccess) e = launch_pdl(spk::k_fc2_reorganize, grid, spk::kFc2Threads, 0, s, p);
  }
  if (e == cudaSuccess) e = cudaGetLastError();
  return e == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

int64_t sp_out_scales_bytes_ex(int64_t T_pad, int64_t H, int quant_mode, int scale_layout) {
  if (T_pad < 0 || H < 0) return -1;
  return scale_bytes_of(T_pad, H, quant_mode, scale_layout);
}

int64_t sp_max_hidden(void) { return kMaxHidden; }

const char* sp_status_string(int status) {
  switch (status) {
    case SP_OK: return "SP_OK";
    case SP_ERR_INVALID_ARG: return "SP_ERR_INVALID_ARG";
    case SP_ERR_UNSUPPORTED: return "SP_ERR_UNSUPPORTED";
    case SP_ERR_ALIGNMENT: return "SP_ERR_ALIGNMENT";
    case SP_ERR_CUDA: return "SP_ERR_CUDA";
    default: return "SP_UNKNOWN_STATUS";
  }
}

sp_status sp_selftest_wait_timeout(uint64_t limit_ns, sp_stream_t stream) {
  if (limit_ns == 0 || limit_ns > spk::kWaitLimitNs) return SP_ERR_INVALID_ARG;
  spk::k_selftest_wait_timeout<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns);
  return cudaGetLastError() == cudaSuccess ? SP_OK : SP_ERR_CUDA;
}

sp_status sp_device_error(uint32_t* flags, int clear) {
  if (!flags) return SP_ERR_INVALID_ARG;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, spk::g_error_flags, sizeof(v)) != cudaSuccess) return SP_ERR_CUDA;
  if (clear) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(spk::g_error_flags, &zero, sizeof(zero)) != cudaSuccess)
      return SP_ERR_CUDA;
  }
  *flags = v;
  return SP_OK;
}

}  // extern "C"

// ------------------------------------------------------------ entry point that allocates nothing
// sp_fused_reduce_norm_noalloc keeps the dynamic row schedule's scratch (its row counter pair) in
// this file's own static device array instead of a per-stream slot or a caller's buffer, so a
// caller that may not allocate device memory still gets that schedule on any stream. The array
// exists once per GPU that loads the library and lives until the process exits.
namespace {

constexpr int kNoAllocScratchWords = 2;  // [next claim, CTAs done]: 8 bytes
// The row counter counts rows with 32-bit atomics on top of the grid; calls with more rows than
// this are refused rather than run with a counter that could wrap.
constexpr int64_t kNoAllocMaxRows = (int64_t{1} << 31) - (int64_t{1} << 16);

static __device__ __align__(256) unsigned int g_noalloc_scratch[kNoAllocScratchWords];

// Device address of g_noalloc_scratch in each device's context, looked up on the first call made
// on that device (with it current). In host code the array's name is only a stand-in for the
// symbol, never a pointer a kernel may be given.
std::atomic<unsigned int*> g_noalloc_scratch_addr[kMaxDevices];
std::mutex g_noalloc_mutex;

sp_status noalloc_scratch(unsigned int** addr) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SP_ERR_CUDA;
  unsigned int* p = g_noalloc_scratch_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    p = g_noalloc_scratch_addr[dev].load(std::memory_order_relaxed);
    if (!p) {
      void* sym = nullptr;
      if (cudaGetSymbolAddress(&sym, g_noalloc_scratch) != cudaSuccess || !sym)
        return SP_ERR_CUDA;
      p = static_cast<unsigned int*>(sym);
      g_noalloc_scratch_addr[dev].store(p, std::memory_order_release);
    }
  }
  *addr = p;
  return SP_OK;
}

}  // namespace

extern "C" {

sp_status sp_fused_reduce_norm_noalloc(const void* partials, int tp, int64_t T_pad,
                                       int64_t T_valid, int64_t H, const void* residual,
                                       const void* weight, const void* bias, float eps,
                                       int quant_mode, const float* scale, void* out,
                                       void* out_scales, void* residual_out,
                                       sp_stream_t stream) {
  sp_status st = check(partials, tp, T_pad, T_valid, H, residual, weight, bias, eps, quant_mode,
                       scale, out, out_scales, residual_out);
  if (st != SP_OK) return st;
  if (T_pad > kNoAllocMaxRows) return SP_ERR_UNSUPPORTED;
  if (T_pad == 0) return SP_OK;
  unsigned int* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != SP_OK) return st;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The array keeps whatever the previous call left: the counter must start at zero.
  if (cudaMemsetAsync(scratch, 0, kNoAllocScratchWords * sizeof(unsigned int), s) != cudaSuccess)
    return SP_ERR_CUDA;
  sp_launch_config cfg;
  st = sp_select_launch(tp, T_pad, H, quant_mode, &cfg);
  if (st != SP_OK) return st;
  Extras x;
  x.row_counter = scratch;
  return run_checked(cfg, partials, tp, T_pad, T_valid, H, residual, weight, bias, eps,
                     quant_mode, scale, out, out_scales, residual_out, s, x);
}

}  // extern "C"
