// Split-KV decode attention on the fifth-generation tensor cores (tcgen05,
// accumulators in tensor memory) for the MQA geometry of "Hand-Writing Gemma 4
// Flash-Decoding + an FP4 Matvec Bonus (Part 2)", section "One KV head breaks
// the textbook": one KV head, up to 16 query rows, head dim 512, bf16 cache,
// no sliding window. Same method as split_tc_kernel (per-split unnormalised
// (O, m, l) partials, one online-softmax rescale per tile, the same merge
// kernel), different machinery:
//
//   * With no window the band is [max(0, len - capacity), len), whose slots
//     are always [0, min(len, capacity)): a split walks slots, not positions,
//     and a tile never wraps the ring (softmax does not depend on order).
//   * Warp 0 streams K and V as TMA tiles (128 positions x 64 head dims,
//     128-byte swizzle, 16 KB) into a ring of 10 chunks; a tile's last, partial
//     rows come in 8-row boxes.
//   * Warp 1 owns the tensor memory and issues the MMAs from one thread:
//     S^T (128 positions x 16 rows, fp32) = K Q^T as 32 MMAs of K = 16 dims,
//     and O^T (512 dims x 16 rows) += V^T P^T as 4 x 8 MMAs per P half, V read
//     MN-major from the same TMA tiles, P = hi + lo bf16 (~16 bits of each
//     weight). The chunks stream as K(0), V(0), K(1), V(1), ...: V(i) lands
//     while the softmax warps work on S(i); S is double-buffered in TMEM.
//   * Warps 2-5 read S from tensor memory (one position per thread), take the
//     row maxima and sums with a halving butterfly (16 shuffles for 16 rows),
//     write P, rescale O in tensor memory when a row's maximum moved, and
//     finally store the partial (or the normalised output when S = 1).
//
// All waits are bounded (fd_device.cuh); the tensor memory is released on
// every path that allocated it.

#include <cuda.h>  // CUtensorMap (descriptor type only; the encoder comes from the runtime)
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cstdint>

#include "fd_decode_attn.h"
#include "fd_internal.h"

namespace fd {
namespace {

#include "fd_device.cuh"

namespace um {
constexpr int HS = 512;                 // head dim
constexpr int NQ = 16;                  // query rows per MMA (N); G <= 16, zero rows above G
constexpr int DC = 64;                  // head dims per chunk: one 128-byte swizzle row
constexpr int NCH = HS / DC;            // chunks per tensor per tile
constexpr int TAIL_ROWS = 8;            // box height for a tile's partial rows
constexpr int NSOFT = 4;                // softmax warps: 2..5, one TMEM lane quarter each
constexpr int THREADS = (2 + NSOFT) * 32;
constexpr int ATOM_Q = NQ * 128;        // 16 rows x 128 B: one K-major swizzle column of Q or P
constexpr int RING_BYTES = 160 * 1024;  // the K/V chunk ring
constexpr uint32_t TMEM_COLS = 128;     // S[2] at columns 0, 16; O block mb at 32 + 16 mb

// Instruction descriptor of tcgen05.mma kind::f16: D f32 (bits 4-5 = 1), A and
// B bf16 (bits 7-9, 10-12 = 1), A MN-major when bit 15 is set, N / 8 at bits
// 17-22, M / 16 at bits 24-28.
constexpr uint32_t idesc_bf16(bool a_mn_major, int M) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         (static_cast<uint32_t>(NQ >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
constexpr uint32_t kIdescPV = idesc_bf16(true, 128);  // A = V^T, MN-major (dims contiguous), M = 128 dims
}  // namespace um

// Tile-dependent layout: T positions per tile (the score MMA's M, 64 or 128).
// An M = 128 accumulator keeps row r in tensor-memory lane r; an M = 64 one
// keeps row r in lane 32 (r / 16) + r % 16 (the first 16 lanes of each
// warp's quarter). P.V always runs with M = 128 head dims.
template <int T_>
struct UmmaTile {
  static constexpr int T = T_;
  static constexpr int CHUNK_BYTES = T * um::DC * 2;             // one TMA box: T positions x 64 dims
  static constexpr int NRING = um::RING_BYTES / CHUNK_BYTES;     // even: a V chunk pair never straddles the wrap
  static constexpr int OFF_RING = 0;
  static constexpr int OFF_Q = OFF_RING + NRING * CHUNK_BYTES;   // Q: NCH atoms of 16 rows x 64 dims
  static constexpr int OFF_P = OFF_Q + um::NCH * um::ATOM_Q;     // P: [2 buffers][hi, lo][T / 64 atoms]
  static constexpr int P_HALF = (T / 64) * um::ATOM_Q;          // T positions of one half (hi or lo)
  static constexpr int P_BUF = 2 * P_HALF;                       // hi + lo
  static constexpr int OFF_RED = OFF_P + 2 * P_BUF;              // f32 [2][NQ][NSOFT] row maxima, row sums
  static constexpr int OFF_BAR = OFF_RED + 2 * um::NQ * um::NSOFT * 4;
  // full[NRING], empty[NRING], q_ready, s_full[2], p_ready[2], pv_done
  static constexpr int NBAR = 2 * NRING + 6;
  static constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;            // u32: tensor memory base address
  static constexpr int SMEM = OFF_TMEM + 16 + 1024;              // + slack to align the base
  static constexpr int LPQ = T / 4;                              // S rows per warp lane quarter
  static constexpr uint32_t kIdescQK = um::idesc_bf16(false, T); // A = K tile, K-major (dims contiguous)

  static_assert(T == 64 || T == 128, "score MMA M");
  static_assert(SMEM <= 227 * 1024, "shared memory");
  static_assert(NRING % 2 == 0 && NRING >= um::NCH, "ring");
  static_assert(OFF_Q % 1024 == 0 && OFF_P % 1024 == 0, "swizzle atoms are 1024-byte aligned");
};

// Positions per tile of the kernel the library launches. Measured on GB300
// (µs per layer, MQA 32k / MQA long at 38 splits): T = 128 26.6 / 189,
// T = 64 35.2 / 321. A tile's time is mostly its fixed chain (softmax, MMA
// commits, P.V before the next scores), so halving the tile doubles it.
constexpr int kUmmaTile = 128;

// Shared-memory matrix descriptor (tcgen05): start address / 16 in bits
// 0-13, leading-dimension byte offset / 16 in 16-29, stride-dimension byte
// offset / 16 in 32-45, descriptor version 1 in 46-47, layout 2 (128-byte
// swizzle) in 61-63. For K-major 128-byte swizzle the rows of an 8-row atom
// are 128 B apart and SBO is the distance between 8-row groups (LBO unused);
// for MN-major, LBO is the distance between 64-element column blocks and SBO
// between 8-row groups along K.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D (tensor memory) = A * B (+ D when accumulate != 0), one thread issues.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The mbarrier gets one arrival when every MMA this thread issued so far has
// completed (and stopped reading its shared-memory operands).
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// 16 consecutive 32-bit columns of this warp's 32 tensor-memory lanes (one
// lane per thread), waited for before returning.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 2-D TMA tile load (x = head dim, y = cache row) completing bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Row reduction of 16 per-thread values (one per query row) over the 32 lanes
// of a warp by halving: each exchange hands half of the rows still held to
// the partner lane, so 8 + 4 + 2 + 1 + 1 shuffles leave lane l with the
// reduction of row l / 2.
template <class Op>
__device__ __forceinline__ float rowreduce16(const float (&v)[16], int lane, Op op) {
  float a8[8], a4[4], a2[2];
  const bool u4 = lane & 16, u3 = lane & 8, u2 = lane & 4, u1 = lane & 2;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    a8[j] = op(u4 ? v[j + 8] : v[j], __shfl_xor_sync(0xffffffffu, u4 ? v[j] : v[j + 8], 16));
#pragma unroll
  for (int j = 0; j < 4; ++j)
    a4[j] = op(u3 ? a8[j + 4] : a8[j], __shfl_xor_sync(0xffffffffu, u3 ? a8[j] : a8[j + 4], 8));
#pragma unroll
  for (int j = 0; j < 2; ++j)
    a2[j] = op(u2 ? a4[j + 2] : a4[j], __shfl_xor_sync(0xffffffffu, u2 ? a4[j] : a4[j + 2], 4));
  const float a1 = op(u1 ? a2[1] : a2[0], __shfl_xor_sync(0xffffffffu, u1 ? a2[0] : a2[1], 2));
  return op(a1, __shfl_xor_sync(0xffffffffu, a1, 1));
}

struct MaxOp {
  __device__ float operator()(float x, float y) const { return fmaxf(x, y); }
};
struct AddOp {
  __device__ float operator()(float x, float y) const { return x + y; }
};

// Chunk stream order shared by the producer and the MMA warp: K(0), V(0),
// K(1), V(1), ... (tensor 0 = K, 1 = V). V(i) streams in while the softmax
// warps work on S(i), so its P.V can start as soon as P(i) is written.
__device__ __forceinline__ void stream_step(int step, int& tensor, int& tile) {
  tensor = step & 1;
  tile = step >> 1;
}

__device__ __forceinline__ void prefetch_tensor_map(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

struct UmmaMaps {
  CUtensorMap k, v;            // boxes of 64 dims x 128 rows
  CUtensorMap k_tail, v_tail;  // boxes of 64 dims x 8 rows
};

template <int T_>
__global__ void __launch_bounds__(um::THREADS, 1)
    split_umma_kernel(const __grid_constant__ UmmaMaps maps, const LaunchArgs a) {
  using namespace um;
  using U = UmmaTile<T_>;
  constexpr int T = U::T, CHUNK_BYTES = U::CHUNK_BYTES, NRING = U::NRING, OFF_RING = U::OFF_RING;
  constexpr int OFF_Q = U::OFF_Q, OFF_P = U::OFF_P, P_HALF = U::P_HALF, P_BUF = U::P_BUF, OFF_RED = U::OFF_RED;
  constexpr int OFF_BAR = U::OFF_BAR, OFF_TMEM = U::OFF_TMEM, LPQ = U::LPQ;
  constexpr uint32_t kIdescQK = U::kIdescQK;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (base - raw);
  const int s = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int G = a.NH / a.NKV;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hbase = kvh * G;

  const uint32_t bar0 = base + OFF_BAR;
  const uint32_t full0 = bar0, empty0 = bar0 + 8 * NRING;
  const uint32_t q_ready = bar0 + 16 * NRING;
  const uint32_t s_full0 = q_ready + 8, p_ready0 = s_full0 + 16, pv_done = p_ready0 + 16;
  float* red = reinterpret_cast<float*>(smem + OFF_RED);

  // Set-up that reads no input, overlapping the previous kernel's tail. The
  // ring starts zeroed: rows past a partial tile then hold zeros or earlier,
  // finite cache rows, and their softmax weight is 0.
  if (tid == 0) {
    for (int k = 0; k < NRING; ++k) {
      mbar_init(full0 + 8 * k, 1);   // the producer's expect_tx arrival + the bytes
      mbar_init(empty0 + 8 * k, 1);  // one tcgen05.commit
    }
    mbar_init(q_ready, NSOFT * 32);
    for (int j = 0; j < 2; ++j) {
      mbar_init(s_full0 + 8 * j, 1);
      mbar_init(p_ready0 + 8 * j, NSOFT * 32);
    }
    mbar_init(pv_done, 1);
    fence_mbar_init();
  }
  if (tid == 32) {
    prefetch_tensor_map(&maps.k);
    prefetch_tensor_map(&maps.v);
    prefetch_tensor_map(&maps.k_tail);
    prefetch_tensor_map(&maps.v_tail);
  }
  for (int i = tid * 16; i < NRING * CHUNK_BYTES; i += THREADS * 16)
    *reinterpret_cast<uint4*>(smem + OFF_RING + i) = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  __syncthreads();  // barriers initialised and the ring zeroed before any copy
  grid_dependency_wait();
  grid_launch_dependents();

  // This split's slots [q0, q0 + n) of the band's slot range [0, band).
  int lo;
  const int band = band_of(a.lens[b], a.capacity, a.window, s == 0 && kvh == 0 && tid == 0, &lo);
  const int chunk = chunk_of(band, a.num_splits, a.granule);
  const long long q0 = static_cast<long long>(s) * chunk;
  const long long q1 = min(static_cast<long long>(band), q0 + chunk);
  const int n = q0 < q1 ? static_cast<int>(q1 - q0) : 0;
  const bool direct = a.num_splits == 1;
  if (n == 0) {  // an empty slice (no TMEM was taken)
    if (direct) {  // len == 0 with one split: the output row is zero
      for (int i = tid; i < G * HS; i += THREADS) {
        const size_t o = (static_cast<size_t>(b) * a.NH + hbase + i / HS) * HS + i % HS;
        a.out[o] = 0;
        if (a.out_f32) a.out_f32[o] = 0.f;
      }
    } else {
      write_empty_partial(a, b, hbase, G, HS, s, tid, THREADS);
    }
    return;
  }
  const int ntiles = (n + T - 1) / T;
  bool failed = false;
  uint32_t tmem = 0;

  if (warp == 0) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      const int row0 = static_cast<int>((static_cast<long long>(b) * a.NKV + kvh) * a.capacity + q0);
      int seq = 0;
      for (int step = 0; step < 2 * ntiles; ++step) {
        int tensor, tile;
        stream_step(step, tensor, tile);
        const int nv = min(T, n - tile * T);
        const int y = row0 + tile * T;
        const CUtensorMap* map = tensor ? (nv == T ? &maps.v : &maps.v_tail) : (nv == T ? &maps.k : &maps.k_tail);
        const int boxes = nv == T ? 1 : (nv + TAIL_ROWS - 1) / TAIL_ROWS;
        const uint32_t box_bytes = nv == T ? CHUNK_BYTES : TAIL_ROWS * 128;
        for (int c = 0; c < NCH; ++c, ++seq) {
          const int slot = seq % NRING, use = seq / NRING;
          if (use > 0) mbar_wait(empty0 + 8 * slot, (use - 1) & 1, failed);
          const uint32_t dst = base + OFF_RING + slot * CHUNK_BYTES;
          const uint32_t fb = full0 + 8 * slot;
          mbar_arrive_expect_tx(fb, boxes * box_bytes);
          for (int r = 0; r < boxes; ++r) tma_load_2d(dst + r * box_bytes, map, c * DC, y + r * TAIL_ROWS, fb);
        }
      }
    }
  } else {
  // The producer needs no tensor memory and starts at once; warps 1-5 wait
  // for warp 1's allocation.
  if (warp == 1) {
    tmem_alloc(base + OFF_TMEM, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  named_bar_sync(3, THREADS - 32);
  tc_fence_after();
  tmem = *reinterpret_cast<const uint32_t*>(smem + OFF_TMEM);

  if (warp == 1) {
    // ------------------------------------------------------- MMA issue warp
    mbar_wait(q_ready, 0, failed);
    tc_fence_after();
    int seq = 0;
    for (int step = 0; step < 2 * ntiles; ++step) {
      int tensor, tile;
      stream_step(step, tensor, tile);
      if (tensor == 0) {
        // S^T(tile) = K Q^T into S buffer tile % 2 (free: the softmax read
        // S(tile - 2) before P(tile - 2) was ready, which P.V(tile - 2) and so
        // this MMA waited for)
        const uint32_t d = tmem + 16 * (tile & 1);
        for (int c = 0; c < NCH; ++c, ++seq) {
          const int slot = seq % NRING;
          mbar_wait(full0 + 8 * slot, (seq / NRING) & 1, failed);
          tc_fence_after();
          if (lane == 0) {
            const uint32_t kb = base + OFF_RING + slot * CHUNK_BYTES;
            const uint32_t qb = base + OFF_Q + c * ATOM_Q;
#pragma unroll
            for (int kk = 0; kk < DC / 16; ++kk)
              umma_bf16(d, sw128_desc(kb + 32 * kk, 16, 1024), sw128_desc(qb + 32 * kk, 16, 1024), kIdescQK,
                        (c | kk) != 0);
            umma_commit(empty0 + 8 * slot);
          }
          __syncwarp();
        }
        if (lane == 0) umma_commit(s_full0 + 8 * (tile & 1));
        __syncwarp();
      } else {
        // O^T += V^T P^T(tile), 128 dims (two chunks) per MMA block
        mbar_wait(p_ready0 + 8 * (tile & 1), (tile >> 1) & 1, failed);
        tc_fence_after();
        const int nv = min(T, n - tile * T);
        const uint32_t pb = base + OFF_P + (tile & 1) * P_BUF;
        for (int mb = 0; mb < NCH / 2; ++mb, seq += 2) {
          const int slot = seq % NRING;  // even: slot + 1 is the pair's second chunk
          mbar_wait(full0 + 8 * slot, (seq / NRING) & 1, failed);
          mbar_wait(full0 + 8 * (slot + 1), ((seq + 1) / NRING) & 1, failed);
          if (nv < T) {
            // rows [nv, nv rounded up to 8) came from slots past the split:
            // zero them (their weight is 0, but they may hold NaN)
            const int r1 = min(T, (nv + TAIL_ROWS - 1) / TAIL_ROWS * TAIL_ROWS);
            const int words = (r1 - nv) * 8;  // 16-byte words per chunk
            for (int w = lane; w < 2 * words; w += 32) {
              const int ch = w / words, rem = w % words;
              *reinterpret_cast<uint4*>(smem + OFF_RING + (slot + ch) * CHUNK_BYTES + (nv + rem / 8) * 128 +
                                        (rem % 8) * 16) = make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
          tc_fence_after();
          if (lane == 0) {
            const uint32_t d = tmem + 32 + 16 * mb;
            const uint32_t vb = base + OFF_RING + slot * CHUNK_BYTES;
#pragma unroll
            for (int kk = 0; kk < T / 16; ++kk) {
              const uint64_t adesc = sw128_desc(vb + kk * 2048, CHUNK_BYTES, 1024);
              const uint32_t patom = pb + (kk >> 2) * ATOM_Q + (kk & 3) * 32;
              umma_bf16(d, adesc, sw128_desc(patom, 16, 1024), kIdescPV, (tile > 0 || kk > 0) ? 1u : 0u);
              umma_bf16(d, adesc, sw128_desc(patom + P_HALF, 16, 1024), kIdescPV, 1u);
            }
            umma_commit(empty0 + 8 * slot);
            umma_commit(empty0 + 8 * (slot + 1));
          }
          __syncwarp();
        }
        if (lane == 0) umma_commit(pv_done);
        __syncwarp();
      }
    }
  } else {
    // ------------------------------------------------- softmax / epilogue warps
    const int sw = warp - 2;             // 0..3
    const int quarter = warp & 3;        // the TMEM lane quarter this warp may access
    const int tq = tid - 64;             // 0..127
    // tile position whose S row this thread's TMEM lane holds (lanes >= LPQ of
    // a quarter hold none when T = 64)
    const bool lane_ok = lane < LPQ;
    const int pl = quarter * LPQ + (lane & (LPQ - 1));
    const uint32_t tlane = static_cast<uint32_t>(quarter * 32) << 16;

    // Q -> shared memory as the K-major, 128-byte-swizzled B operand: atom c
    // holds dims [64 c, 64 c + 64) of the 16 rows; rows >= G are zero.
    {
      constexpr int kPer = NQ * HS / 8 / (NSOFT * 32);  // 16-byte pieces per thread
      uint4 v[kPer];
#pragma unroll
      for (int k = 0; k < kPer; ++k) {  // every load in flight before the first store
        const int id = tq + k * NSOFT * 32, r = id / (HS / 8), dc = id % (HS / 8);
        v[k] = r < G ? *reinterpret_cast<const uint4*>(a.q + (static_cast<size_t>(b) * a.NH + hbase + r) * HS + dc * 8)
                     : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int k = 0; k < kPer; ++k) {
        const int id = tq + k * NSOFT * 32, r = id / (HS / 8), dc = id % (HS / 8), j = dc % 8;
        *reinterpret_cast<uint4*>(smem + OFF_Q + (dc / 8) * ATOM_Q + (r / 8) * 1024 + (r % 8) * 128 +
                                  ((j ^ (r % 8)) * 16)) = v[k];
      }
    }
    fence_proxy_async_smem();
    mbar_arrive(q_ready);

    float m_run[NQ], l_run[NQ];
#pragma unroll
    for (int r = 0; r < NQ; ++r) {
      m_run[r] = kNegInf;
      l_run[r] = 0.f;
    }
    for (int i = 0; i < ntiles; ++i) {
      const int nv = min(T, n - i * T);
      mbar_wait(s_full0 + 8 * (i & 1), (i >> 1) & 1, failed);
      tc_fence_after();
      float sc[NQ];
      tmem_ld16(tmem + tlane + 16 * (i & 1), sc);
      const bool valid = lane_ok && pl < nv;
#pragma unroll
      for (int r = 0; r < NQ; ++r) sc[r] = valid ? sc[r] * a.scale_log2 : kNegInf;

      // row maxima of the tile: warp butterfly, then the four warps' values
      const float wmax = rowreduce16(sc, lane, MaxOp());
      if ((lane & 1) == 0) red[(lane >> 1) * NSOFT + sw] = wmax;
      named_bar_sync(2, NSOFT * 32);
      float m_new[NQ], alpha[NQ], p[NQ];
#pragma unroll
      for (int r = 0; r < NQ; ++r) {
        const float4 t = *reinterpret_cast<const float4*>(red + r * NSOFT);
        m_new[r] = fmaxf(m_run[r], fmaxf(fmaxf(t.x, t.y), fmaxf(t.z, t.w)));
        alpha[r] = m_new[r] == kNegInf ? 1.f : exp2f(m_run[r] - m_new[r]);
        p[r] = m_new[r] == kNegInf ? 0.f : exp2f(sc[r] - m_new[r]);
      }

      // P = hi + lo bf16 -> buffer i % 2, K-major and swizzled like Q (its
      // last reader, P.V(i - 2), finished before tile i - 1 released its P)
      {
        unsigned char* pbuf = smem + OFF_P + (i & 1) * P_BUF + (pl >> 6) * ATOM_Q;
        const int pc = (pl & 63) >> 3, pw = (pl & 7) * 2;
        if (lane_ok) {
#pragma unroll
          for (int r = 0; r < NQ; ++r) {
            const uint16_t hi = f32_to_bf16_bits(p[r]);
            const uint16_t lo = f32_to_bf16_bits(p[r] - bf16_bits_to_f32(hi));
            unsigned char* at = pbuf + (r >> 3) * 1024 + (r & 7) * 128 + ((pc ^ (r & 7)) << 4) + pw;
            *reinterpret_cast<uint16_t*>(at) = hi;
            *reinterpret_cast<uint16_t*>(at + P_HALF) = lo;
          }
        }
      }

      // row sums
      const float wsum = rowreduce16(p, lane, AddOp());
      if ((lane & 1) == 0) red[NQ * NSOFT + (lane >> 1) * NSOFT + sw] = wsum;
      named_bar_sync(2, NSOFT * 32);
      bool moved = false;
#pragma unroll
      for (int r = 0; r < NQ; ++r) {
        const float4 t = *reinterpret_cast<const float4*>(red + NQ * NSOFT + r * NSOFT);
        l_run[r] = l_run[r] * alpha[r] + ((t.x + t.y) + (t.z + t.w));
        moved |= alpha[r] != 1.f;
      }

      // O *= alpha in tensor memory once P.V(i - 1) is done (every thread
      // holds the same alphas, so the branch is uniform)
      if (i > 0) {
        mbar_wait(pv_done, (i - 1) & 1, failed);
        tc_fence_after();
        if (moved) {
#pragma unroll
          for (int mb = 0; mb < NCH / 2; ++mb) {
            float o[NQ];
            tmem_ld16(tmem + tlane + 32 + 16 * mb, o);
#pragma unroll
            for (int r = 0; r < NQ; ++r) o[r] *= alpha[r];
            tmem_st16(tmem + tlane + 32 + 16 * mb, o);
          }
          tmem_st_wait();
        }
      }
#pragma unroll
      for (int r = 0; r < NQ; ++r) m_run[r] = m_new[r];
      fence_proxy_async_smem();  // P stores -> the tensor cores' view of shared memory
      tc_fence_before();
      mbar_arrive(p_ready0 + 8 * (i & 1));
    }

    // ---- epilogue: this thread's dim of each 128-dim block, all rows
    mbar_wait(pv_done, (ntiles - 1) & 1, failed);
    tc_fence_after();
#pragma unroll
    for (int mb = 0; mb < NCH / 2; ++mb) {
      float o[NQ];
      tmem_ld16(tmem + tlane + 32 + 16 * mb, o);
      const int d = mb * 128 + quarter * 32 + lane;  // O^T lanes are head dims
#pragma unroll
      for (int r = 0; r < NQ; ++r) {
        if (r >= G) break;
        const size_t row = static_cast<size_t>(b) * a.NH + hbase + r;
        if (direct) {
          const float x = o[r] / l_run[r];
          a.out[row * HS + d] = f32_to_bf16_bits(x);
          if (a.out_f32) a.out_f32[row * HS + d] = x;
        } else {
          a.ws_o[(row * a.num_splits + s) * HS + d] = o[r];
        }
      }
    }
    if (!direct && tq < G) {
      const size_t row = static_cast<size_t>(b) * a.NH + hbase + tq;
      float mr = m_run[0], lr = l_run[0];
#pragma unroll
      for (int r = 1; r < NQ; ++r)
        if (r == tq) {
          mr = m_run[r];
          lr = l_run[r];
        }
      a.ws_ml[(row * a.num_splits + s) * 2 + 0] = mr;
      a.ws_ml[(row * a.num_splits + s) * 2 + 1] = lr;
    }
  }
  }

  // release the tensor memory once every warp is done with it
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// The cache [B * NKV * capacity rows][512 dims] as a 2-D bf16 tensor with
// 128-byte swizzled boxes of 64 dims x `rows`.
bool encode_cache_map(CUtensorMap* m, const void* base, const LaunchArgs& a, uint32_t rows) {
  const auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(um::HS),
                              static_cast<cuuint64_t>(a.B) * a.NKV * static_cast<cuuint64_t>(a.capacity)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(um::HS) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(um::DC), rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool umma_shape_ok(int HS, int G, int window) { return HS == um::HS && G > 8 && G <= um::NQ && window <= 0; }

cudaError_t launch_umma(const LaunchArgs& a, cudaStream_t stream) {
  if (!umma_shape_ok(a.HS, a.NH / a.NKV, a.window) || a.cluster != 1 || a.fused || a.kv8 ||
      static_cast<long long>(a.B) * a.NKV * a.capacity >= (1ll << 31))
    return cudaErrorInvalidValue;
  UmmaMaps maps;
  if (!encode_cache_map(&maps.k, a.k, a, kUmmaTile) || !encode_cache_map(&maps.v, a.v, a, kUmmaTile) ||
      !encode_cache_map(&maps.k_tail, a.k, a, um::TAIL_ROWS) || !encode_cache_map(&maps.v_tail, a.v, a, um::TAIL_ROWS))
    return cudaErrorInvalidValue;
  constexpr int kSmem = UmmaTile<kUmmaTile>::SMEM;
  cudaError_t e =
      cudaFuncSetAttribute(split_umma_kernel<kUmmaTile>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.num_splits, a.NKV, a.B);
  cfg.blockDim = dim3(um::THREADS);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, split_umma_kernel<kUmmaTile>, maps, a);
}

cudaError_t set_wait_limit_umma(unsigned long long ns) {
  const unsigned long long v = ns ? ns : 1000000000ull;
  return cudaMemcpyToSymbol(g_wait_limit_ns, &v, sizeof v);
}

cudaError_t read_and_clear_device_error_umma(unsigned int* err) {
  unsigned int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof v);
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
  *err |= v;
  return e;
}

}  // namespace fd
