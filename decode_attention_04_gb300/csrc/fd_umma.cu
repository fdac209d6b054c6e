// Split-KV decode attention on the fifth-generation tensor cores (tcgen05,
// accumulators in tensor memory) for the MQA geometry of "Hand-Writing Gemma 4
// Flash-Decoding + an FP4 Matvec Bonus (Part 2)", section "One KV head breaks
// the textbook": one KV head, up to 16 query rows, head dim 512, bf16 cache,
// no sliding window. Same method as split_tc_kernel (per-split unnormalised
// (O, m, l) partials merged by the same merge kernels), different machinery:
//
//   * With no window the band is [max(0, len - capacity), len), whose slots
//     are always [0, min(len, capacity)): a split takes the consecutive slots
//     [s * chunk, (s + 1) * chunk) of that range (the softmax does not depend
//     on the order of positions), in tiles of 128.
//   * Warp 0 streams K and V as TMA boxes (128-byte swizzle, 64 head dims
//     wide) through one ring of 32 KB slots, each a pair of chunks (128
//     positions x 128 dims: one P.V MMA block, or two K chunks). The stream
//     order is K(0), then V(i) and K(i + 1) pair by pair, then the last
//     tile's V: V(i) is requested while K(i + 1) streams, so it lands about
//     when P(i) is ready instead of holding slots through the softmax, and
//     the scores of tile i + 1 never wait for V. Boxes are 128, 64, 32, 16
//     or 8 rows high, so a tile's rows are read exactly; the last rows of a
//     slice that do not fill 8 are loaded by the copy warp's lanes and stored
//     into the same swizzled layout. Nothing outside the band is read.
//   * Warp 1 owns the tensor memory and issues every MMA from one thread, out
//     of order between two streams: S^T (128 positions x 16 rows, fp32) =
//     K Q^T as each K chunk lands (4 MMAs of K = 16 dims per chunk, into one
//     of two S buffers), and O^T (512 dims x 16 rows) += V^T P^T for tile i
//     once P(i) is ready and each V pair lands (P = hi + lo bf16, ~16 bits of
//     each weight). The scores of tile i + 1 are therefore computed while the
//     softmax of tile i runs, and the K stream never waits for V.
//   * Warps 2-5 read S from tensor memory (one position per thread), take the
//     tile's row maxima with a halving butterfly (16 shuffles for 16 rows) and
//     one barrier, and write P. The running maximum moves only when a row's
//     tile maximum exceeds it by more than 2^8 (then O is rescaled in tensor
//     memory once the previous P.V is done); otherwise the weights, at most
//     2^8, are taken against the old maximum, which gives the same softmax.
//     Row sums stay per thread until the end: one reduction per split.
//
// All waits are bounded (fd_device.cuh); the copy warp waits for its last
// copies and the MMA warp for its last MMAs before the block leaves, and the
// tensor memory is released on every path that allocated it.

#include <cuda.h>  // CUtensorMap (descriptor type only; the encoder comes from the runtime)
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <atomic>
#include <cstdint>
#include <mutex>

#include "fd_decode_attn.h"
#include "fd_internal.h"

namespace fd {
namespace {

#include "fd_device.cuh"

namespace um {
constexpr int HS = 512;                   // head dim
constexpr int NQ = 16;                    // query rows per MMA (N); G <= 16, zero rows above G
constexpr int T = 128;                    // positions per tile: the score MMA's M
constexpr int DC = 64;                    // head dims per chunk: one 128-byte swizzle row
constexpr int NCH = HS / DC;              // chunks per tensor per tile
constexpr int CHUNK_BYTES = T * DC * 2;   // one 128-row TMA box: 16 KB
constexpr int PAIR_BYTES = 2 * CHUNK_BYTES;  // 128 positions x 128 dims: one ring slot
constexpr int NPAIR = NCH / 2;            // pairs per tensor per tile
constexpr int NPS = 6;                    // ring slots (pairs), K and V alike
constexpr int MAX_TAIL = (NCH * 7 * 8 + 31) / 32;  // 16-byte tail pieces per lane (a tile's tensor, at most 7 rows)
constexpr int NMAP = 5;                   // box heights T, T/2, T/4, T/8, T/16 (= 8)
constexpr int NSOFT = 4;                  // softmax warps, one TMEM lane quarter each
constexpr int W_COPY = 0, W_MMA = 1, W_SOFT0 = 2;
constexpr int THREADS = (W_SOFT0 + NSOFT) * 32;
constexpr int ATOM_Q = NQ * 128;          // 16 rows x 128 B: one K-major swizzle column of Q or P
constexpr int P_HALF = (T / 64) * ATOM_Q; // T positions of one half (hi or lo)
constexpr int P_BUF = 2 * P_HALF;         // hi + lo
constexpr int OFF_RING = 0;
constexpr int OFF_Q = OFF_RING + NPS * PAIR_BYTES;  // Q: NCH atoms of 16 rows x 64 dims
constexpr int OFF_P = OFF_Q + NCH * ATOM_Q;         // P: [2 buffers][hi, lo][T / 64 atoms]
constexpr int OFF_RED = OFF_P + 2 * P_BUF;          // f32 [2][NQ][NSOFT] tile maxima, [NQ][NSOFT] sums
constexpr int RED_FLOATS = 3 * NQ * NSOFT;
constexpr int OFF_BAR = OFF_RED + RED_FLOATS * 4;
// full[NPS], empty[NPS], s_full[2], s_free[2], p_ready[2], pv_done[2], q_ready, mma_done
constexpr int NBAR = 2 * NPS + 8 + 2;
constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;      // u32: tensor memory base address
constexpr int SMEM = OFF_TMEM + 16 + 1024;        // + slack to align the base to 1024
constexpr uint32_t TMEM_COLS = 128;               // S[2] at columns 0, 16; O block mb at 32 + 16 mb
constexpr float kRescaleLog2 = 8.f;               // the running max moves when a tile's exceeds it by 2^8

static_assert(SMEM <= 227 * 1024, "shared memory");
static_assert(OFF_Q % 1024 == 0 && OFF_P % 1024 == 0, "swizzle atoms are 1024-byte aligned");
static_assert((T >> (NMAP - 1)) == 8, "smallest box: 8 rows (1024 bytes, one swizzle atom)");
static_assert(MAX_TAIL * 32 >= NCH * 7 * 8, "every tail piece of a tile's tensor has a lane");

// The one copy stream: K(0), then V(i) and K(i + 1) pair by pair, then the
// last tile's V. Stream position of each pair (ring slot = position % NPS).
__device__ __forceinline__ int seq_k(int t, int p) { return t == 0 ? p : NPAIR + 2 * NPAIR * (t - 1) + 2 * p + 1; }
__device__ __forceinline__ int seq_v(int t, int p, int ntiles) {
  return NPAIR + 2 * NPAIR * t + (t + 1 < ntiles ? 2 * p : p);
}

// Instruction descriptor of tcgen05.mma kind::f16: D f32 (bits 4-5 = 1), A and
// B bf16 (bits 7-9, 10-12 = 1), A MN-major when bit 15 is set, N / 8 at bits
// 17-22, M / 16 at bits 24-28.
constexpr uint32_t idesc_bf16(bool a_mn_major, int M) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         (static_cast<uint32_t>(NQ >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
constexpr uint32_t kIdescQK = idesc_bf16(false, T);   // A = K tile, K-major (dims contiguous), M = 128 positions
constexpr uint32_t kIdescPV = idesc_bf16(true, 128);  // A = V^T, MN-major (dims contiguous), M = 128 dims
}  // namespace um

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

// Transaction bytes a phase of the barrier will receive, without an arrival
// (the arrival comes after the copy warp's own stores into the same stage).
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// 2-D TMA tile load (x = head dim, y = cache row) completing bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void prefetch_tensor_map(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
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

struct UmmaMaps {
  CUtensorMap k[um::NMAP], v[um::NMAP];  // boxes of 64 dims x 128, 64, 32, 16, 8 rows
};

__global__ void __launch_bounds__(um::THREADS, 1)
    split_umma_kernel(const __grid_constant__ UmmaMaps maps, const LaunchArgs a) {
  using namespace um;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* smem = smem_raw + (base - raw);
  const int s = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int S = a.num_splits;
  const int G = a.NH / a.NKV;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hbase = kvh * G;

  const uint32_t bar0 = base + OFF_BAR;
  const uint32_t full = bar0, empty = full + 8 * NPS;
  const uint32_t s_full = empty + 8 * NPS, s_free = s_full + 16, p_ready = s_free + 16, pv_done = p_ready + 16;
  const uint32_t q_ready = pv_done + 16, mma_done = q_ready + 8;
  float* red = reinterpret_cast<float*>(smem + OFF_RED);

  // Set-up that reads no input, overlapping the previous kernel's tail.
  if (tid == 0) {
    for (int k = 0; k < NPS; ++k) {
      mbar_init(full + 8 * k, 1);   // the copy warp's arrival + the bytes
      mbar_init(empty + 8 * k, 1);  // one tcgen05.commit
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(s_full + 8 * j, 1);
      mbar_init(s_free + 8 * j, NSOFT * 32);
      mbar_init(p_ready + 8 * j, NSOFT * 32);
      mbar_init(pv_done + 8 * j, 1);
    }
    mbar_init(q_ready, NSOFT * 32);
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  if (warp == W_COPY && lane < 2 * NMAP) prefetch_tensor_map(lane < NMAP ? &maps.k[lane] : &maps.v[lane - NMAP]);
  __syncthreads();
  grid_dependency_wait();
  grid_launch_dependents();

  // This split's slots [q0, q0 + n) of the band's slot range [0, band).
  const int len_b = a.lens[b];
  const bool reporter = s == 0 && kvh == 0 && tid == 0;
  if (reporter && len_b < a.min_len) atomicOr(&g_device_error, FD_DEVERR_MIN_LEN);
  int lo;
  const int band = band_of(len_b, a.capacity, a.window, reporter, &lo);
  const int chunk = chunk_of(band, S, a.granule);
  const long long q0 = static_cast<long long>(s) * chunk;
  const int n = q0 < band ? static_cast<int>(min(static_cast<long long>(chunk), band - q0)) : 0;
  const bool direct = S == 1;
  if (n == 0) {  // an empty slice: no copy issued, no tensor memory taken
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
  const int row0 = static_cast<int>((static_cast<long long>(b) * a.NKV + kvh) * a.capacity + q0);
  bool failed = false;

  // The MMA warp allocates the tensor memory; it and the softmax warps meet
  // before using it. The copy warp needs none and starts at once.
  uint32_t tmem = 0;
  if (warp >= W_MMA) {
    if (warp == W_MMA) {
      tmem_alloc(base + OFF_TMEM, TMEM_COLS);
      tmem_relinquish();
    }
    tc_fence_before();
    named_bar_sync(2, (1 + NSOFT) * 32);
    tc_fence_after();
    tmem = *reinterpret_cast<const uint32_t*>(smem + OFF_TMEM);
  }

  if (warp == W_COPY) {
    // ------------------------------------------------------------ copy warp
    // One stream of 32 KB pairs (128 positions x 128 dims) through one ring:
    // K(0), then V(i) and K(i + 1) alternately, then the last tile's V. V(i)
    // is requested while K(i + 1) streams, so it lands about when P(i) is
    // ready instead of holding slots through the softmax, and the scores of
    // tile i + 1 never wait for V.
    uint32_t st_issued = 0, st_par = 0;
    const int total = 2 * NPAIR * ntiles;
    // The rows of the slice's last tile that do not fill 8 (its only partial
    // tile) come from the lanes: all of a tensor's pieces of that tile are
    // loaded at its first pair, in one round trip, and stored pair by pair.
    // K of the last tile is done before its V starts, so one array serves.
    uint4 tailv[MAX_TAIL];
    for (int e = 0; e < total; ++e) {
      bool is_k;
      int t, pr;
      if (e < NPAIR) {
        is_k = true, t = 0, pr = e;
      } else {
        const int m = e - NPAIR, i = m / (2 * NPAIR), r = m % (2 * NPAIR);
        if (i + 1 < ntiles) {
          is_k = r & 1, pr = r >> 1, t = is_k ? i + 1 : i;
        } else {
          is_k = false, pr = r, t = i;
        }
      }
      const CUtensorMap* mp = is_k ? maps.k : maps.v;
      const uint16_t* src = is_k ? a.k : a.v;
      const int nv = min(T, n - t * T);
      const int nv8 = nv & ~7;      // rows the TMA boxes bring
      const int nrem = nv - nv8;    // the slice's last rows: loaded by the lanes
      const int y0 = row0 + t * T;  // cache row of the tile's first position
      if (nrem > 0 && pr == 0) {
#pragma unroll
        for (int k = 0; k < MAX_TAIL; ++k) {  // piece i: chunk i / (8 nrem), row nv8 + (i / 8) % nrem, piece i % 8
          const int i = lane + 32 * k;
          tailv[k] = make_uint4(0, 0, 0, 0);
          if (i < NCH * nrem * 8) {
            const int c = i / (nrem * 8), rr = nv8 + (i / 8) % nrem, j = i % 8;
            tailv[k] = *reinterpret_cast<const uint4*>(src + static_cast<size_t>(y0 + rr) * HS + c * DC + j * 8);
          }
        }
      }
      const int slot = e % NPS, use = e / NPS;
      if (use > 0) mbar_wait(empty + 8 * slot, (use - 1) & 1, failed);
      const uint32_t dst = base + OFF_RING + slot * PAIR_BYTES;
      const uint32_t fb = full + 8 * slot;
      unsigned char* dsts = smem + (dst - base);
      if (lane == 0) {
        mbar_expect_tx(fb, static_cast<uint32_t>(2 * nv8) * 128);
        for (int h = 0; h < 2; ++h) {
          const int c = 2 * pr + h;
          const uint32_t d = dst + h * CHUNK_BYTES;
          if (nv8 == T) {
            tma_load_2d(d, &mp[0], c * DC, y0, fb);
          } else {
            int r = 0;
#pragma unroll
            for (int bi = 1; bi < NMAP; ++bi) {
              const int bh = T >> bi;
              if (nv8 & bh) {
                tma_load_2d(d + r * 128, &mp[bi], c * DC, y0 + r, fb);
                r += bh;
              }
            }
          }
        }
      }
      const int nz = ((nv + 15) & ~15) - nv;  // V rows the last 16-row P.V step reads past the tile
      if (!is_k && nz > 0) {
        // zero them, so their 0 weights add exactly 0 (stale shared memory may
        // hold any bit pattern). P.V reads no row past that step, and with
        // 16-position chunks only a split ending at the band's end has any.
        const int words = nz * (DC * 2 / 16);  // 16-byte words per chunk
        for (int w = lane; w < 2 * words; w += 32) {
          const int ch = w / words, rem = w % words;
          *reinterpret_cast<uint4*>(dsts + ch * CHUNK_BYTES + (nv + rem / 8) * 128 + (rem % 8) * 16) =
              make_uint4(0, 0, 0, 0);
        }
      }
      if (nrem > 0) {
        // this pair's pieces, into the 128-byte swizzle (piece j of row r
        // sits at 16 * (j ^ (r % 8)))
#pragma unroll
        for (int k = 0; k < MAX_TAIL; ++k) {
          const int i = lane + 32 * k;
          const int c = i / (nrem * 8);
          if (i < NCH * nrem * 8 && (c >> 1) == pr) {
            const int rr = nv8 + (i / 8) % nrem, j = i % 8;
            *reinterpret_cast<uint4*>(dsts + (c & 1) * CHUNK_BYTES + rr * 128 + ((j ^ (rr & 7)) << 4)) = tailv[k];
          }
        }
      }
      if (nrem > 0 || (!is_k && nz > 0)) fence_proxy_async_smem();  // lanes' stores -> the tensor cores' view
      __syncwarp();
      if (lane == 0) mbar_arrive(fb);
      st_issued |= 1u << slot;
      st_par = (st_par & ~(1u << slot)) | (static_cast<uint32_t>(use & 1) << slot);
    }
    // No copy of this block may still be in flight when it leaves: wait for
    // the last phase issued into each slot (bounded, own failure flag).
    bool dfail = false;
    for (int k = 0; k < NPS; ++k)
      if ((st_issued >> k) & 1u) mbar_wait(full + 8 * k, (st_par >> k) & 1u, dfail);
  } else if (warp == W_MMA) {
    // ----------------------------------------------------- MMA issue thread
    if (lane == 0) {
      mbar_wait(q_ready, 0, failed);
      tc_fence_after();
      int kt = 0, kp = 0;  // next score MMAs: tile kt, K pair kp
      int vt = 0, vp = 0;  // next P.V MMAs: tile vt, V pair (128-dim block) vp
      bool s_ok = false, p_ok = false;
      uint64_t t_idle = 0;
      uint32_t spins = 0;  // polls without progress; the clock is read every 4096
      while ((kt < ntiles || vt < ntiles) && !failed) {
        bool prog = false;
        if (kt < ntiles) {
          // S buffer kt % 2 is free once the softmax has read S(kt - 2)
          if (!s_ok) s_ok = kt < 2 || mbar_test(s_free + 8 * (kt & 1), ((kt - 2) >> 1) & 1);
          const int e = seq_k(kt, kp), slot = e % NPS;
          if (s_ok && mbar_test(full + 8 * slot, (e / NPS) & 1)) {
            tc_fence_after();
            const uint32_t kb = base + OFF_RING + slot * PAIR_BYTES;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int c = 2 * kp + h;
              const uint32_t qb = base + OFF_Q + c * ATOM_Q;
#pragma unroll
              for (int kk = 0; kk < DC / 16; ++kk)
                umma_bf16(tmem + 16 * (kt & 1), sw128_desc(kb + h * CHUNK_BYTES + 32 * kk, 16, 1024),
                          sw128_desc(qb + 32 * kk, 16, 1024), kIdescQK, (c | kk) != 0);
            }
            umma_commit(empty + 8 * slot);
            if (++kp == NPAIR) {
              umma_commit(s_full + 8 * (kt & 1));
              kp = 0;
              ++kt;
              s_ok = false;
            }
            prog = true;
          }
        }
        if (vt < kt) {
          if (!p_ok) p_ok = mbar_test(p_ready + 8 * (vt & 1), (vt >> 1) & 1);
          const int e = seq_v(vt, vp, ntiles), slot = e % NPS;
          if (p_ok && mbar_test(full + 8 * slot, (e / NPS) & 1)) {
            tc_fence_after();
            const uint32_t vb = base + OFF_RING + slot * PAIR_BYTES;
            const uint32_t pb = base + OFF_P + (vt & 1) * P_BUF;
            const uint32_t d = tmem + 32 + 16 * vp;
            const int nk = (min(T, n - vt * T) + 15) >> 4;  // 16-position steps holding valid rows
            for (int kk = 0; kk < nk; ++kk) {
              const uint64_t adesc = sw128_desc(vb + kk * 2048, CHUNK_BYTES, 1024);
              const uint32_t patom = pb + (kk >> 2) * ATOM_Q + (kk & 3) * 32;
              umma_bf16(d, adesc, sw128_desc(patom, 16, 1024), kIdescPV, (vt > 0 || kk > 0) ? 1u : 0u);
              umma_bf16(d, adesc, sw128_desc(patom + P_HALF, 16, 1024), kIdescPV, 1u);
            }
            umma_commit(empty + 8 * slot);
            if (++vp == NPAIR) {
              umma_commit(pv_done + 8 * (vt & 1));
              vp = 0;
              ++vt;
              p_ok = false;
            }
            prog = true;
          }
        }
        if (prog) {
          spins = 0;
        } else if ((++spins & 4095u) == 0) {
          const uint64_t now = globaltimer_ns();
          if (spins == 4096u) {
            t_idle = now;
          } else if (now - t_idle > g_wait_limit_ns) {
            failed = true;
            atomicOr(&g_device_error, FD_DEVERR_WAIT_TIMEOUT);
          }
        }
      }
      // every MMA issued has completed before the block can release the
      // tensor memory
      umma_commit(mma_done);
      bool dfail = false;
      mbar_wait(mma_done, 0, dfail);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------- softmax / epilogue warps
    const int sw = warp - W_SOFT0;  // 0..3
    const int quarter = warp & 3;   // the TMEM lane quarter this warp may access
    const int tq = tid - W_SOFT0 * 32;
    const int pl = quarter * 32 + lane;  // tile position whose S row this thread's TMEM lane holds
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

    float m_use[NQ], l_part[NQ];  // reference maxima (log2 units); this thread's share of the row sums
#pragma unroll
    for (int r = 0; r < NQ; ++r) {
      m_use[r] = kNegInf;
      l_part[r] = 0.f;
    }
    for (int i = 0; i < ntiles; ++i) {
      const int nv = min(T, n - i * T);
      mbar_wait(s_full + 8 * (i & 1), (i >> 1) & 1, failed);
      tc_fence_after();
      float sc[NQ];
      tmem_ld16(tmem + tlane + 16 * (i & 1), sc);
      tc_fence_before();
      mbar_arrive(s_free + 8 * (i & 1));  // S(i) read: its buffer may take S(i + 2)
      const bool valid = pl < nv;
#pragma unroll
      for (int r = 0; r < NQ; ++r) sc[r] = valid ? sc[r] * a.scale_log2 : kNegInf;

      // the tile's row maxima: warp butterfly, then the four warps' values
      float* rm = red + (i & 1) * NQ * NSOFT;
      const float wmax = rowreduce16(sc, lane, MaxOp());
      if ((lane & 1) == 0) rm[(lane >> 1) * NSOFT + sw] = wmax;
      named_bar_sync(1, NSOFT * 32);
      bool resc = false;
      float alpha[NQ];
#pragma unroll
      for (int r = 0; r < NQ; ++r) {
        const float4 t4 = *reinterpret_cast<const float4*>(rm + r * NSOFT);
        const float mt = fmaxf(fmaxf(t4.x, t4.y), fmaxf(t4.z, t4.w));
        const bool need = mt > m_use[r] + kRescaleLog2;  // false for -inf and NaN tile maxima
        alpha[r] = need ? exp2f(m_use[r] - mt) : 1.f;
        if (need) m_use[r] = mt;
        resc |= need;
      }
      // every thread took the same decision from the same shared values
      if (resc) {
#pragma unroll
        for (int r = 0; r < NQ; ++r) l_part[r] *= alpha[r];
        if (i > 0) {  // O holds P.V of the earlier tiles: rescale it once P.V(i - 1) is done
          mbar_wait(pv_done + 8 * ((i - 1) & 1), ((i - 1) >> 1) & 1, failed);
          tc_fence_after();
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
      float p[NQ];
#pragma unroll
      for (int r = 0; r < NQ; ++r) {
        p[r] = exp2f(sc[r] - m_use[r]);
        l_part[r] += p[r];
      }

      // P = hi + lo bf16 -> buffer i % 2, K-major and swizzled like Q; its
      // last reader, P.V(i - 2), must be done
      if (i >= 2) mbar_wait(pv_done + 8 * (i & 1), ((i - 2) >> 1) & 1, failed);
      {
        unsigned char* pbuf = smem + OFF_P + (i & 1) * P_BUF + (pl >> 6) * ATOM_Q;
        const int pc = (pl & 63) >> 3, pw = (pl & 7) * 2;
#pragma unroll
        for (int r = 0; r < NQ; ++r) {
          const uint16_t hi = f32_to_bf16_bits(p[r]);
          const uint16_t lo16 = f32_to_bf16_bits(p[r] - bf16_bits_to_f32(hi));
          unsigned char* at = pbuf + (r >> 3) * 1024 + (r & 7) * 128 + ((pc ^ (r & 7)) << 4) + pw;
          *reinterpret_cast<uint16_t*>(at) = hi;
          *reinterpret_cast<uint16_t*>(at + P_HALF) = lo16;
        }
      }
      fence_proxy_async_smem();  // P stores -> the tensor cores' view of shared memory
      tc_fence_before();
      mbar_arrive(p_ready + 8 * (i & 1));
    }

    // ---- epilogue: the row sums, then this thread's dim of each 128-dim block
    float* rs = red + 2 * NQ * NSOFT;
    const float lsum = rowreduce16(l_part, lane, AddOp());
    if ((lane & 1) == 0) rs[(lane >> 1) * NSOFT + sw] = lsum;
    named_bar_sync(1, NSOFT * 32);
    float L[NQ];
#pragma unroll
    for (int r = 0; r < NQ; ++r) {
      const float4 t4 = *reinterpret_cast<const float4*>(rs + r * NSOFT);
      L[r] = (t4.x + t4.y) + (t4.z + t4.w);  // fixed order
    }
    mbar_wait(pv_done + 8 * ((ntiles - 1) & 1), ((ntiles - 1) >> 1) & 1, failed);
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
          const float x = o[r] / L[r];
          a.out[row * HS + d] = f32_to_bf16_bits(x);
          if (a.out_f32) a.out_f32[row * HS + d] = x;
        } else {
          a.ws_o[(row * S + s) * HS + d] = o[r];
        }
      }
    }
    if (!direct && tq < G) {
      float mr = m_use[0], lr = L[0];
#pragma unroll
      for (int r = 1; r < NQ; ++r)
        if (r == tq) {
          mr = m_use[r];
          lr = L[r];
        }
      const size_t row = static_cast<size_t>(b) * a.NH + hbase + tq;
      reinterpret_cast<float2*>(a.ws_ml)[row * S + s] = make_float2(mr, lr);
    }
  }

  // release the tensor memory once every warp is done with it
  tc_fence_before();
  __syncthreads();
  if (warp == W_MMA) {
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

// A cache [rows][512 dims] as a 2-D bf16 tensor with 128-byte swizzled boxes
// of 64 dims x `box_rows`.
bool encode_cache_map(CUtensorMap* m, const void* base, long long rows, uint32_t box_rows) {
  const auto enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(um::HS), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(um::HS) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(um::DC), box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Encoded maps of recent (K, V, rows) caches: encoding ten maps costs several
// microseconds of host time, and a decode loop calls with the same caches
// every step. Direct-mapped by the K address.
struct MapEntry {
  const void* k = nullptr;
  const void* v = nullptr;
  long long rows = 0;
  UmmaMaps maps;
};
constexpr int kMapCache = 128;
std::mutex g_map_mu;
MapEntry g_map_cache[kMapCache];

bool cached_maps(const LaunchArgs& a, UmmaMaps* out) {
  const long long rows = static_cast<long long>(a.B) * a.NKV * a.capacity;
  const size_t slot = (reinterpret_cast<uintptr_t>(a.k) >> 12) % kMapCache;
  std::lock_guard<std::mutex> lk(g_map_mu);
  MapEntry& e = g_map_cache[slot];
  if (e.k != a.k || e.v != a.v || e.rows != rows) {
    UmmaMaps m;
    for (int i = 0; i < um::NMAP; ++i) {
      const uint32_t h = static_cast<uint32_t>(um::T >> i);
      if (!encode_cache_map(&m.k[i], a.k, rows, h) || !encode_cache_map(&m.v[i], a.v, rows, h)) return false;
    }
    e.k = a.k;
    e.v = a.v;
    e.rows = rows;
    e.maps = m;
  }
  *out = e.maps;
  return true;
}

}  // namespace

bool umma_shape_ok(int HS, int G, int window) { return HS == um::HS && G > 8 && G <= um::NQ && window <= 0; }

int umma_tile_positions() { return um::T; }

cudaError_t launch_umma(const LaunchArgs& a, cudaStream_t stream) {
  if (!umma_shape_ok(a.HS, a.NH / a.NKV, a.window) || a.cluster != 1 || a.fused || a.kv8 ||
      static_cast<long long>(a.B) * a.NKV * a.capacity >= (1ll << 31))
    return cudaErrorInvalidValue;
  UmmaMaps maps;
  if (!cached_maps(a, &maps)) return cudaErrorInvalidValue;
  static std::atomic<unsigned long long> attr_done{0};  // bit d: attribute set on device d
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (bit == 0 || (attr_done.load(std::memory_order_acquire) & bit) == 0) {
    e = cudaFuncSetAttribute(split_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, um::SMEM);
    if (e != cudaSuccess) return e;
    attr_done.fetch_or(bit, std::memory_order_acq_rel);
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.num_splits, a.NKV, a.B);
  cfg.blockDim = dim3(um::THREADS);
  cfg.dynamicSmemBytes = um::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, split_umma_kernel, maps, a);
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
