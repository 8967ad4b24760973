// Shared device helpers of the sm_103a routed-MoE library.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "moe.h"

namespace moe {

// ---------------------------------------------------------------------------
// Record geometry: gate | up | down | gate_s | up_s | down_s, K contiguous.
// ---------------------------------------------------------------------------
struct RecordOffsets {
  size_t gate, up, down, gate_s, up_s, down_s, total;
};

__host__ __device__ inline int block_elems(int fmt) { return fmt == MOE_FMT_NVFP4 ? 16 : 32; }

__host__ __device__ inline RecordOffsets record_offsets(int H, int I, int fmt) {
  RecordOffsets o;
  const size_t codes = (size_t)I * (size_t)H / 2;
  const size_t scales = (size_t)I * (size_t)H / (size_t)block_elems(fmt);
  o.gate = 0;
  o.up = codes;
  o.down = 2 * codes;
  o.gate_s = 3 * codes;
  o.up_s = 3 * codes + scales;
  o.down_s = 3 * codes + 2 * scales;
  o.total = 3 * codes + 3 * scales;
  return o;
}

inline bool shape_ok(const moe_expert_shape& s) {
  return s.hidden > 0 && s.inter > 0 && s.hidden % 64 == 0 && s.inter % 64 == 0 &&
         s.hidden <= 16384 && s.inter <= 8192 &&
         (s.format == MOE_FMT_NVFP4 || s.format == MOE_FMT_MXFP4);
}

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

inline int launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

// ---------------------------------------------------------------------------
// Per-device facts and kernel attributes.  A process may drive several GPUs
// (one per thread, or one after another), so everything that depends on the
// device -- its SM count, its shared-memory limit, and the dynamic
// shared-memory size a kernel was allowed on it -- is kept per device id.
// ---------------------------------------------------------------------------
constexpr int kMaxDevices = 64;

inline std::mutex& host_mutex() {
  static std::mutex m;
  return m;
}

inline int current_device() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}

struct DeviceInfo {
  int sms;         // streaming multiprocessors
  int smem_optin;  // largest dynamic shared memory one block may opt in to
};

// The current device's facts, looked up once per device; {0, 0} when there
// is no usable device.
inline DeviceInfo device_info() {
  static std::atomic<int> sms[kMaxDevices], smem[kMaxDevices];
  const int d = current_device();
  if (d < 0) return DeviceInfo{0, 0};
  int a = sms[d].load(std::memory_order_acquire);
  if (a == 0) {
    std::lock_guard<std::mutex> lock(host_mutex());
    int n = 0, m = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&m, cudaDevAttrMaxSharedMemoryPerBlockOptin, d) != cudaSuccess)
      return DeviceInfo{0, 0};
    smem[d].store(m, std::memory_order_relaxed);
    sms[d].store(n, std::memory_order_release);
    a = n;
  }
  return DeviceInfo{a, smem[d].load(std::memory_order_relaxed)};
}

// Dynamic shared memory granted to one kernel, per device.
struct SmemGrant {
  std::atomic<size_t> bytes[kMaxDevices];
};

// Raises `kernel`'s dynamic shared-memory limit on the current device to
// `bytes` unless an earlier call already did; the attribute call is made once
// per (kernel, device, size increase), so later launches can be captured in
// a graph.  With `threads` > 0 the kernel runs a grid-wide barrier over one
// CTA per SM, which needs every CTA resident at once: the grant then also
// checks that one CTA of `threads` threads and `bytes` bytes fits on an SM
// (it returns false otherwise).  Kernels of other streams, processes (MPS) or
// green contexts that hold SMs can still keep CTAs waiting; the barrier waits
// are bounded and report MOE_DEV_TIMEOUT then.
template <typename K>
inline bool grant_smem(K kernel, size_t bytes, SmemGrant& g, int threads = 0) {
  const int d = current_device();
  if (d < 0) return false;
  const size_t key = bytes + 1;  // 0 means "nothing checked yet", also for small sizes
  if (key <= g.bytes[d].load(std::memory_order_acquire)) return true;
  std::lock_guard<std::mutex> lock(host_mutex());
  if (key <= g.bytes[d].load(std::memory_order_relaxed)) return true;
  if (bytes > 48 * 1024 &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) != cudaSuccess)
    return false;
  if (threads > 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, bytes) != cudaSuccess || n < 1)
      return false;
  }
  g.bytes[d].store(key, std::memory_order_release);
  return true;
}

// ---------------------------------------------------------------------------
// Scalar conversions
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

// BF16 x BF16 + FP32 with one rounding, on the low halves of the words: both
// factors are exact in FP32, so the result is the FP32 FMA of the converted
// values, without converting them first.
__device__ __forceinline__ float fma_bf16(uint32_t a_lo16, uint32_t b_lo16, float c) {
  float d;
  asm("fma.rn.f32.bf16 %0, %1, %2, %3;"
      : "=f"(d)
      : "h"((uint16_t)(a_lo16 & 0xFFFFu)), "h"((uint16_t)(b_lo16 & 0xFFFFu)), "f"(c));
  return d;
}

// Two E4M3 bytes (low byte = first) -> two floats, via the hardware convert.
__device__ __forceinline__ float2 e4m3x2_to_f32x2(uint32_t two_bytes) {
  uint32_t h2;
  uint16_t in = (uint16_t)(two_bytes & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
  __half2 hh = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(hh);
}

// UE8M0 byte -> 2^(s-127) as float (s = 0 is the subnormal 2^-127, 255 NaN).
__device__ __forceinline__ float ue8m0_to_f32(uint32_t s) {
  s &= 0xFFu;
  if (s == 0xFFu) return __uint_as_float(0x7FC00000u);
  if (s == 0u) return __uint_as_float(0x00400000u);
  return __uint_as_float(s << 23);
}

// One byte of two e2m1 codes -> f16x2 (low nibble -> low half).
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte_in_low8) {
  uint32_t h2;
  asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}"
      : "=r"(h2)
      : "r"(byte_in_low8));
  return h2;
}

// Packed FP32 FMA: (d.x, d.y) = (a.x * b.x + c.x, a.y * b.y + c.y).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  unsigned long long ra, rb, rc, rd;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rc) : "f"(c.x), "f"(c.y));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  float2 d;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
  return d;
}

// 16-byte load of weights read once: no L1 allocation, and the L2 fetches the
// surrounding 256 bytes so the following k-steps of the same row hit in L2.
__device__ __forceinline__ uint4 ldg_stream_l2pf(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Streaming 16-byte load that does not allocate in L1 (weights are read once).
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Sum over 8 e2m1 codes of one 32-bit word times 8 consecutive floats of xs
// (xs 8-byte aligned); two running sums in acc.
__device__ __forceinline__ float2 dot8_e2m1(uint32_t w, const float* xs, float2 acc) {
#pragma unroll
  for (int b = 0; b < 4; ++b) {
    uint32_t h2 = e2m1x2_to_f16x2((w >> (8 * b)) & 0xFFu);
    float2 wf = __half22float2(*reinterpret_cast<__half2*>(&h2));
    float2 xv = *reinterpret_cast<const float2*>(xs + 2 * b);
    acc = ffma2(wf, xv, acc);
  }
  return acc;
}

// One 16-byte unit of codes (32 elements) dotted with xs[0..31] and scaled by
// its block scale(s): NVFP4 has two E4M3 scales (elements 0-15, 16-31), MXFP4
// one UE8M0 scale.  `sbits` holds the scale byte(s), first block in the low byte.
template <int FMT>
__device__ __forceinline__ float unit_dot(uint4 q, uint32_t sbits, const float* xs) {
  float2 a = make_float2(0.f, 0.f), b = make_float2(0.f, 0.f);
  a = dot8_e2m1(q.x, xs + 0, a);
  a = dot8_e2m1(q.y, xs + 8, a);
  b = dot8_e2m1(q.z, xs + 16, b);
  b = dot8_e2m1(q.w, xs + 24, b);
  if (FMT == MOE_FMT_NVFP4) {
    float2 s = e4m3x2_to_f32x2(sbits);
    return (a.x + a.y) * s.x + (b.x + b.y) * s.y;
  } else {
    return ((a.x + a.y) + (b.x + b.y)) * ue8m0_to_f32(sbits);
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int d = 16; d > 0; d >>= 1) v += __shfl_xor_sync(0xffffffffu, v, d);
  return v;
}

__device__ __forceinline__ void status_or(int32_t* st, int bits) {
  if (st) atomicOr(st, bits);
}

}  // namespace moe

namespace moe {

// Programmatic dependent launch: let the next kernel in the stream start its
// prologue now, and wait until the previous kernel's results are visible.
// Both are no-ops for a kernel launched without the PDL attribute.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ unsigned ld_acquire_gpu(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier for a grid whose CTAs are all resident (one CTA per SM,
// checked on the host before the launch).  bar[0] counts arrivals and is reset to 0 by the last arriver,
// bar[1] is an epoch that the last arriver bumps; the others wait for the
// epoch to move, at most until `deadline_ns`.  bar[0] must be 0 before the
// first use and is 0 again after every completed barrier.  Returns false
// (for every thread of the CTA) if the wait ran out.
__device__ __forceinline__ bool grid_barrier(unsigned* bar, unsigned nblocks, uint64_t deadline_ns,
                                             int* smem_flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    const unsigned e0 = ld_acquire_gpu(bar + 1);
    __threadfence();
    const unsigned old = atomicAdd(bar, 1u);
    if (old == nblocks - 1) {
      atomicExch(bar, 0u);
      __threadfence();
      atomicAdd(bar + 1, 1u);
    } else {
      while (ld_acquire_gpu(bar + 1) == e0) {
        if (global_ns() > deadline_ns) {
          ok = 0;
          break;
        }
      }
    }
    __threadfence();
    *smem_flag = ok;
  }
  __syncthreads();
  return *smem_flag != 0;
}

}  // namespace moe

namespace moe {

// Launches `kernel` with programmatic stream serialization, so it may start
// while the previous kernel on the stream is finishing; the kernel itself
// calls pdl_wait() before touching anything the previous kernel produced.
// With `cooperative`, the launch is also cooperative: the driver runs it only
// with every CTA resident at once (else the launch fails), which a kernel
// with a grid-wide barrier needs.
template <typename... KArgs, typename... Args>
inline int launch_pdl_ex(bool cooperative, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                         cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeCooperative;
  attr[1].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cooperative ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

template <typename... KArgs, typename... Args>
inline int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t stream, Args... args) {
  return launch_pdl_ex(false, kernel, grid, block, smem, stream, args...);
}

}  // namespace moe
