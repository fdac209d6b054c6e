// Device-side helpers shared by the split kernels (fd_kernels.cu, fd_umma.cu):
// the band and chunk rules, bf16 bit conversions, mbarrier waits that give up
// after about a second, bulk copies, programmatic dependent launch, cluster
// and proxy fences. Included inside `namespace fd { namespace { ... } }`, so
// every translation unit gets its own copy, including its own device error
// word `g_device_error` (read back by that unit's host code).
#pragma once

__device__ unsigned int g_device_error;

// Wall-time limit of every bounded wait, nanoseconds (about one second; the
// host may shorten it for a test of the timeout path).
__device__ unsigned long long g_wait_limit_ns = 1000000000ull;

constexpr float kNegInf = -__builtin_huge_valf();

// Live band of sequence b: positions [lo, lo + band). Reports repaired
// lengths through the device error word when `report` is set.
__device__ __forceinline__ int band_of(int len, int capacity, int window, bool report, int* lo) {
  unsigned flags = 0;
  if (len < 0) {
    flags |= FD_DEVERR_LEN_NEGATIVE;
    len = 0;
  }
  int keep = capacity;
  if (window > 0) {
    keep = min(window, capacity);
  } else if (len > capacity) {
    flags |= FD_DEVERR_LEN_CLAMPED;
  }
  const int l0 = max(0, len - keep);
  if (report && flags) atomicOr(&g_device_error, flags);
  *lo = l0;
  return len - l0;
}

// Positions per split for a band: ceil(band / S) rounded up to the granule.
__device__ __forceinline__ int chunk_of(int band, int num_splits, int granule) {
  const long long c = (static_cast<long long>(band) + num_splits - 1) / num_splits;
  const long long r = ((c + granule - 1) / granule) * granule;
  return static_cast<int>(r < granule ? granule : r);
}

__device__ __forceinline__ int active_splits(int band, int chunk) {
  return band <= 0 ? 0 : (band + chunk - 1) / chunk;
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t h) {
  return __uint_as_float(static_cast<uint32_t>(h) << 16);
}

__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// The partial of a split whose slice of the band is empty: O = 0, m = -inf,
// l = 0, which has weight 0 in the merge. Every split block writes one, so the
// merge kernel reads all S partial slots of a row without first reading the
// row's length. G rows of HS floats at slot s of S; HS % 4 == 0.
__device__ __forceinline__ void write_empty_partial(const LaunchArgs& a, int b, int hbase, int G, int HS, int s,
                                                    int tid, int nthreads) {
  const int S = a.num_splits;
  const int hs4 = HS / 4;
  for (int i = tid; i < G * hs4; i += nthreads) {
    const size_t row = static_cast<size_t>(b) * a.NH + hbase + i / hs4;
    reinterpret_cast<float4*>(a.ws_o + (row * S + s) * HS)[i % hs4] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int g = tid; g < G; g += nthreads) {
    const size_t row = static_cast<size_t>(b) * a.NH + hbase + g;
    reinterpret_cast<float2*>(a.ws_ml)[row * S + s] = make_float2(kNegInf, 0.f);
  }
}

// ------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of a phase (try_wait may suspend the thread for a while
// when the phase is not complete; a thread that polls several barriers, or
// only asks whether data has landed yet, must move on at once).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait: gives up after g_wait_limit_ns of wall time (about one
// second) past its first 256 polls, raises FD_DEVERR_WAIT_TIMEOUT and returns
// false. `failed` is sticky
// per thread, so after one timeout every later wait of that thread returns at
// once and the kernel runs to its end; no wait in this library can hang the
// GPU.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, bool& failed) {
  if (failed) return false;
  // The clock is read only every 256 unsuccessful polls (a wait that ends
  // soon never reads it); the limit counts from the first reading.
  uint64_t t0 = 0;
  for (uint32_t i = 0;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u) {
      const uint64_t now = globaltimer_ns();
      if (i == 255u) {
        t0 = now;
      } else if (now - t0 > g_wait_limit_ns) {
        break;
      }
    }
  }
  failed = true;
  atomicOr(&g_device_error, FD_DEVERR_WAIT_TIMEOUT);
  return false;
}

// 1-D bulk async copy global -> this CTA's shared memory, completing bytes on
// the mbarrier. dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Hint: bring [p, p + bytes) into L2 (no data reaches the thread; p and
// bytes multiples of 16). A later load still reads whatever L2 then holds, so
// the hint may precede a wait for the kernel that writes those bytes.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Programmatic dependent launch: a kernel launched with
// cudaLaunchAttributeProgrammaticStreamSerialization may start while the
// previous kernel on the stream is still running. It must wait for that
// kernel (and its memory) before reading any input; it lets the next kernel
// launch once every one of its own blocks has started. Both are no-ops for a
// kernel launched without the attribute.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Thread-block clusters: rank of this block in its cluster, another block's
// shared-memory address, loads through distributed shared memory, and a
// barrier over every thread of the cluster (release/acquire, so shared-memory
// writes before it are visible to the whole cluster after it).
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t map_to_rank(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}

__device__ __forceinline__ float ld_dsmem(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ float4 ld_dsmem4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

