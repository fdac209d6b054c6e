// Split-KV decode attention kernels for sm_103a (GB300).
//
// The method is the Flash-Decoding formulation of "Hand-Writing Gemma 4
// Flash-Decoding + an FP4 Matvec Bonus (Part 2)", section "One KV head breaks
// the textbook": every (sequence b, KV head, split s) thread block takes its
// share of the live band [max(0, len - W), len), reads position p from cache
// slot p % capacity, and leaves an unnormalised (O, m, l) partial; a merge
// kernel combines the partials with the online-softmax rule. Softmax state is
// rescaled once per tile of positions, not once per position (same section,
// last bullet).
//
// Kernels:
//   split_simt_kernel  per-position fp32 kernel; the plain reference GPU path.
//   split_tc_kernel    the hot path: a producer warp streams K/V rows of the
//                      band into a ring of shared-memory stages with 1-D bulk
//                      async copies (cp.async.bulk + mbarrier transaction
//                      counts); consumer warps compute the Q-group scores of a
//                      tile with bf16 tensor-core MMAs (S^T = K Q^T, so the
//                      positions fill the 16-row side and the G <= 16 query
//                      rows the 8-wide side), rescale once per tile, and
//                      accumulate O^T = V^T P^T on the tensor cores.
//   merge_kernel       online-softmax merge of the S partials of each row
//                      (few rows); merge_staged_kernel, the same for many rows,
//                      with the partials brought into shared memory.

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <type_traits>
#include <utility>

#include "fd_decode_attn.h"
#include "fd_internal.h"

namespace fd {
namespace {

#include "fd_device.cuh"

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A(16x16, row) * B(16x8, col), bf16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D += A(16x16, row) * B(16x8, col), fp16 operands, fp32 accumulators.
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two E4M3 codes (low byte = first element) to an fp16 pair (low half = first),
// exactly: every E4M3 value, subnormals included, is an fp16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t codes) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(codes), __NV_E4M3);
  return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  return static_cast<uint32_t>(__half_as_ushort(__float2half_rn(lo))) |
         (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(hi))) << 16);
}

// ======================================================= SIMT reference kernel

constexpr int kSimtThreads = 128;

// One block per (split, KV head, sequence). Each thread owns dims
// tid, tid + 128, ... of every query row of the group; per position the G dot
// products are reduced across the block, the online-softmax state is updated
// for that single position, and O is rescaled. Shared memory: q [G][HS],
// O [G][HS], per-warp partial dots [4][G], and per-row m, l, alpha, p.
__global__ void __launch_bounds__(kSimtThreads) split_simt_kernel(const LaunchArgs a) {
  extern __shared__ float sm[];
  const int s = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int G = a.NH / a.NKV, HS = a.HS;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float* sq = sm;                    // [G][HS]
  float* so = sq + G * HS;           // [G][HS]
  float* sred = so + G * HS;         // [4][G]
  float* sm_run = sred + 4 * G;      // [G]
  float* sl_run = sm_run + G;        // [G]
  float* salpha = sl_run + G;        // [G]
  float* sp = salpha + G;            // [G]

  grid_dependency_wait();
  grid_launch_dependents();
  int lo;
  const int band = band_of(a.lens[b], a.capacity, a.window, s == 0 && kvh == 0 && tid == 0, &lo);
  const int chunk = chunk_of(band, a.num_splits, a.granule);
  const long long p0 = lo + static_cast<long long>(s) * chunk;
  const long long p1 = min(static_cast<long long>(lo) + band, p0 + chunk);
  const bool direct = a.num_splits == 1;
  const int hbase = kvh * G;

  if (p0 >= p1) {
    if (direct) {  // len == 0: the output row is zero
      for (int i = tid; i < G * HS; i += kSimtThreads) {
        const size_t o = (static_cast<size_t>(b) * a.NH + hbase + i / HS) * HS + i % HS;
        a.out[o] = 0;
        if (a.out_f32) a.out_f32[o] = 0.f;
      }
    } else {
      write_empty_partial(a, b, hbase, G, HS, s, tid, kSimtThreads);
    }
    return;
  }

  for (int i = tid; i < G * HS; i += kSimtThreads) {
    sq[i] = bf16_bits_to_f32(a.q[(static_cast<size_t>(b) * a.NH + hbase) * HS + i]);
    so[i] = 0.f;
  }
  if (tid < G) {
    sm_run[tid] = kNegInf;
    sl_run[tid] = 0.f;
  }
  __syncthreads();

  const size_t head_row0 = (static_cast<size_t>(b) * a.NKV + kvh) * a.capacity;
  for (long long pos = p0; pos < p1; ++pos) {
    const size_t row = (head_row0 + static_cast<size_t>(pos % a.capacity)) * HS;
    for (int g = 0; g < G; ++g) {
      float part = 0.f;
      for (int d = tid; d < HS; d += kSimtThreads) part += sq[g * HS + d] * bf16_bits_to_f32(a.k[row + d]);
      for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
      if (lane == 0) sred[warp * G + g] = part;
    }
    __syncthreads();
    if (tid < G) {
      float sc = 0.f;
      for (int w = 0; w < kSimtThreads / 32; ++w) sc += sred[w * G + tid];
      sc *= a.scale_log2;
      const float m_old = sm_run[tid];
      const float m_new = fmaxf(m_old, sc);
      const float alpha = (m_new == kNegInf) ? 1.f : exp2f(m_old - m_new);
      const float p = exp2f(sc - m_new);
      sl_run[tid] = sl_run[tid] * alpha + p;
      sm_run[tid] = isnan(sc) ? sc : m_new;
      salpha[tid] = isnan(sc) ? sc : alpha;
      sp[tid] = p;
    }
    __syncthreads();
    for (int g = 0; g < G; ++g) {
      const float al = salpha[g], p = sp[g];
      for (int d = tid; d < HS; d += kSimtThreads)
        so[g * HS + d] = so[g * HS + d] * al + p * bf16_bits_to_f32(a.v[row + d]);
    }
  }
  __syncthreads();

  for (int i = tid; i < G * HS; i += kSimtThreads) {
    const int g = i / HS, d = i % HS;
    const int h = hbase + g;
    if (direct) {
      const float val = so[i] / sl_run[g];
      const size_t o = (static_cast<size_t>(b) * a.NH + h) * HS + d;
      a.out[o] = f32_to_bf16_bits(val);
      if (a.out_f32) a.out_f32[o] = val;
    } else {
      a.ws_o[((static_cast<size_t>(b) * a.NH + h) * a.num_splits + s) * HS + d] = so[i];
    }
  }
  if (!direct && tid < G) {
    const size_t r = ((static_cast<size_t>(b) * a.NH + hbase + tid) * a.num_splits + s) * 2;
    a.ws_ml[r] = sm_run[tid];
    a.ws_ml[r + 1] = sl_run[tid];
  }
}

size_t simt_smem_bytes(int G, int HS) {
  return (static_cast<size_t>(2) * G * HS + 4 * G + 4 * G) * sizeof(float);
}

// ===================================================== tensor-core split kernel

// Shared-memory staging of a tile. The K (and V) rows of a tile arrive as NG
// groups of R consecutive positions, GROUP_BYTES (2 or 4 KB) per group, so one
// bulk copy moves a whole group: a block's copy rate is set by the number of
// copies it issues (on GB300, about 15 / 23 / 33 / 45 GB/s per block with
// 0.5 / 1 / 2 / 4 KB copies), not by their bytes. Groups are 16 bytes apart
// beyond their R rows. Row i of group g holds tile position g*R + i.
//
// The MMAs walk the tile in a permuted order: MMA row m takes group m % NG,
// row m / NG. Eight consecutive MMA rows then sit in eight different groups,
// i.e. in eight different 16-byte bank groups, so every 8-row ldmatrix is
// conflict-free. Scores, P and the P.V contraction all use the same order;
// the softmax does not depend on the order of positions.
//
// E4M3 caches (KV8): the ring holds the codes in 1 KB groups (the same tile
// positions as the bf16 tile, half the bytes), and the consumers build fp16
// MMA fragments from it in registers. The order of the k index of an MMA is
// free as long as both operands use the same one, so for S^T = K Q^T a
// thread's four k slots are four consecutive head dims (one 32-bit load per
// K row); for O^T = V^T P^T the k slots are MMA rows as usual and a
// thread's 32-bit load holds four consecutive dims of one position, which
// byte permutes split into the rows of two MMAs: accumulator row grp of
// MMA 2c holds dim 32c + 4 grp, row grp + 8 dim 32c + 4 grp + 1, and MMA
// 2c + 1 the dims + 2 and + 3. With the 16-byte group padding both load
// patterns are free of bank conflicts.
template <int HS_, int NT_, int NWC_, int NSTAGE_, int GROUP_BYTES_ = 2048, bool KV8_ = false, int MAXREG_ = 0>
struct TcCfg {
  static constexpr bool KV8 = KV8_;
  static constexpr int HS = HS_;
  static constexpr int NT = NT_;          // 8-row tiles of query rows (G <= 8 * NT)
  static constexpr int NP = 8 * NT;       // padded query rows
  static constexpr int NWC = NWC_;        // consumer warps
  static constexpr int NSTAGE = NSTAGE_;  // shared-memory ring depth
  static constexpr int ROWB = HS * 2;     // bytes of one cache row
  static constexpr int R = ROWB >= GROUP_BYTES_ ? 1 : GROUP_BYTES_ / ROWB;  // rows per group
  static constexpr int NG = 8;            // groups per tile
  static constexpr int T = NG * R;        // positions per pipeline tile
  static constexpr int GP = R * ROWB + 16;  // group pitch, bytes
  static constexpr int THREADS = (NWC + 2) * 32;  // consumers + a K and a V producer warp
  static constexpr int CTHREADS = NWC * 32;
  static constexpr int DW = HS / NWC;     // head dims owned by one consumer warp
  static constexpr int KD = DW / 16;      // 16-dim steps per warp
  static constexpr int MP = T / 16;       // 16-row MMA tiles per pipeline tile
  static constexpr int PPITCH = T + 8;    // P row pitch (bf16)
  static constexpr int TPR = CTHREADS / NP;  // softmax threads per query row
  // E4M3 tiles with at most NP / 2 real query rows: twice the threads per row
  // (one warp at most) and half the positions each, so the softmax skips the
  // padded rows and each warp reads one row of scores (no bank conflicts).
  // Measured on GB300 (us per layer): E4M3 Llama ragged 152.3 -> 140.8,
  // tiny 5.70 -> 5.62; the bf16 tiles lost (ragged 159.4 -> 163.2), so they
  // keep the full mapping. Head dim 512 keeps it too: its tiles serve 16-row
  // MQA groups, and the second mapping compiled into them alone cost E4M3
  // MQA long 123.6 -> 128.3 and MQA 32k 21.7 -> 22.5.
  static constexpr int TPR2 =
      (KV8 && HS <= 256 && 2 * TPR <= 32 && T % (2 * TPR) == 0) ? 2 * TPR : TPR;
  static constexpr size_t STAGE_BYTES = static_cast<size_t>(NG) * GP;
  // bf16 tiles held: the copy ring itself, or none (KV8 reads its own ring)
  static constexpr int NBUF = KV8 ? 0 : NSTAGE;
  static constexpr int ROWB8 = HS;                // bytes of one E4M3 cache row
  static constexpr int GP8 = R * ROWB8 + 16;      // E4M3 group pitch, bytes
  static constexpr size_t STAGE8_BYTES = KV8 ? static_cast<size_t>(NG) * GP8 : 0;
  static constexpr size_t OFF_K = 0;
  static constexpr size_t OFF_V = OFF_K + NBUF * STAGE_BYTES;
  static constexpr size_t OFF_K8 = OFF_V + NBUF * STAGE_BYTES;   // E4M3 copy ring (KV8 only)
  static constexpr size_t OFF_V8 = OFF_K8 + NSTAGE * STAGE8_BYTES;
  static constexpr int SP = T + 4;       // score row pitch (floats): conflict-free stores and loads
  static constexpr size_t OFF_S = OFF_V8 + NSTAGE * STAGE8_BYTES;            // f32 [NWC][NP][SP]
  static constexpr size_t OFF_P = OFF_S + static_cast<size_t>(NWC) * NP * SP * 4;  // bf16 [2][NP][PPITCH]
  static constexpr size_t OFF_A = OFF_P + static_cast<size_t>(2) * NP * PPITCH * 2;  // f32 alpha,m,l [NP]
  static constexpr size_t OFF_BAR = (OFF_A + 3 * NP * 4 + 7) / 8 * 8;        // u64 full[], empty[]
  static constexpr size_t SMEM = OFF_BAR + 2 * NSTAGE * 8;
  // blocks per SM the shared memory allows (two when a block takes at most
  // half of the SM's 228 KB, less the 1 KB the driver reserves per block);
  // the in-launch merge instances are held to it by a register bound (the plain
  // instance is left to the compiler, which keeps it leaner)
  static constexpr int MINB = SMEM + 1024 <= 114 * 1024 ? 2 : 1;
  // Register budget of the plain per-split instance (0: the compiler's
  // choice, under launch bounds only), set where a measurement depends on it
  // (GB300, us per layer): a tile meant to run two blocks per SM must fit
  // twice (the bf16 MQA tile at 106 registers ran one block per SM, two
  // waves: 212 against 164 for MQA long), and the one-block-per-SM MQA tiles
  // ran best at 96 (E4M3 MQA 32k 22.5 at 119 registers, 21.7 at 96). A
  // budget given to every instance slowed others (E4M3 MQA long 122 -> 144),
  // so only these configurations take one. Where one-tile splits wait for the
  // merge kernel, that kernel's blocks must fit beside two split blocks (the
  // ring tile at 82 registers, where none fits, 7.0; the compiler's choice
  // without the fused merge in the instance, 6.1). The in-launch merge
  // instances are held by their launch bounds to the occupancy their shared
  // memory allows (the group step needs every block resident at once).
  static constexpr int MAXREG = MAXREG_;

  // tile position held by MMA row m, and its byte offset in a stage
  __device__ static __forceinline__ int pos_of(int m) { return (m % NG) * R + m / NG; }
  __device__ static __forceinline__ int off_of(int m) { return (m % NG) * GP + (m / NG) * ROWB; }
  // byte offset of tile position j in a stage
  __device__ static __forceinline__ int off_pos(int j) { return (j / R) * GP + (j % R) * ROWB; }
  // byte offset of MMA row m in an E4M3 stage
  __device__ static __forceinline__ int off8_of(int m) { return (m % NG) * GP8 + (m / NG) * ROWB8; }
  // head dim (within the warp's slice) of accumulator row grp (+ 8 when hi) of dim-MMA mt
  __device__ static __forceinline__ int dim_of(int mt, int grp, int hi) {
    return KV8 ? 32 * (mt >> 1) + 4 * grp + 2 * (mt & 1) + hi : mt * 16 + grp + hi * 8;
  }
  // smallest tile position among MMA rows [16 mt, 16 mt + 16)
  __device__ static __forceinline__ int min_pos(int mt) { return pos_of(16 * mt); }

  static_assert(HS % (16 * NWC) == 0, "head dims must split into 16-wide slices per warp");
  static_assert(NG % 8 == 0, "eight consecutive MMA rows must fall in eight groups");
  static_assert(T % 16 == 0 && T % TPR == 0, "tile must be whole 16-position MMA tiles");
  static_assert(TPR <= 32 && 32 % TPR == 0, "a row's softmax threads must sit in one warp");
  static_assert(ROWB % 16 == 0 && GP % 16 == 0, "bulk copies need 16-byte granules");
  static_assert(NG <= 32, "one producer lane per group");
  // cluster reduction: O parked in the tile buffers (all of [0, OFF_S) is idle
  // once the last tile is consumed), weights in the score buffer
  static_assert(static_cast<size_t>(NP) * HS * 4 <= OFF_S, "O must fit the tile buffers");
  static_assert(!KV8 || (GP8 % 16 == 0 && (R * ROWB8 == 1024 || R * ROWB8 == 2048)),
                "E4M3 groups are 1 or 2 KB, 16-byte aligned");
  static_assert(!KV8 || DW % 32 == 0, "E4M3 fragments take head dims 32 at a time");
  static_assert(NP * 16 + 2 * NP <= NWC * NP * SP, "cluster weights must fit the score buffer");
};

constexpr int kLptMaxB = 64;
constexpr int kItemQ = 4;  // work items a persistent block's roles may be apart

// Order in which the split blocks (or a persistent grid's work items) visit
// the sequences: s_seq[z] = the z-th longest band (ties by index) when
// 1 < B <= kLptMaxB, else the identity (s_seq unused). Blocks start in
// blockIdx order and work items are taken in index order, so the longest
// splits start first and the last wave holds the short ones
// (longest-processing-time-first order); every order gives the same partials.
__device__ __forceinline__ bool lpt_ordered(const LaunchArgs& a) { return a.B > 1 && a.B <= kLptMaxB; }

__device__ void lpt_table(const LaunchArgs& a, int tid, int nthreads, int* s_seq) {
  if (!lpt_ordered(a)) return;
  int lo;
  for (int t = tid; t < a.B; t += nthreads) {
    const int bt = band_of(a.lens[t], a.capacity, a.window, false, &lo);
    int rank = 0;
    for (int u = 0; u < a.B; ++u) {
      const int bu = band_of(a.lens[u], a.capacity, a.window, false, &lo);
      rank += (bu > bt) || (bu == bt && u < t);
    }
    s_seq[rank] = t;
  }
}

// Source bytes of one producer warp's tensor (K for the first producer warp,
// V for the second) for (sequence b, KV head kvh), and its stage ring offset.
template <class C>
__device__ __forceinline__ const unsigned char* producer_src(const LaunchArgs& a, bool is_k, int b, int kvh) {
  const size_t head_row0 = (static_cast<size_t>(b) * a.NKV + kvh) * a.capacity;
  return C::KV8 ? (is_k ? a.k8 : a.v8) + head_row0 * C::HS
                : reinterpret_cast<const unsigned char*>((is_k ? a.k : a.v) + head_row0 * C::HS);
}

template <class C>
__device__ __forceinline__ size_t producer_ring(bool is_k) {
  return C::KV8 ? (is_k ? C::OFF_K8 : C::OFF_V8) : (is_k ? C::OFF_K : C::OFF_V);
}

// The bulk copies of one pipeline tile of one tensor: positions
// [pbase, pbase + nv) (slot = position mod capacity) into stage st; lane g
// copies group g (rows [g*R, g*R + rows) of the tile) and every lane arrives
// on the stage's full barrier with the bytes it copies.
template <class C>
__device__ __forceinline__ void produce_tile(const LaunchArgs& a, const unsigned char* src, uint32_t stage_dst,
                                             uint32_t fb, long long pbase, int nv, int lane) {
  constexpr int kRowBytes = C::KV8 ? C::ROWB8 : C::ROWB;
  constexpr int kGroupPitch = C::KV8 ? C::GP8 : C::GP;
  const int g = lane;
  const int j0 = g * C::R;
  const int rows = (g < C::NG && j0 < nv) ? min(C::R, nv - j0) : 0;
  mbar_arrive_expect_tx(fb, static_cast<uint32_t>(rows) * kRowBytes);
  if (rows > 0) {
    const long long pos0 = pbase + j0;
    const size_t slot0 = static_cast<size_t>(pos0 % a.capacity);
    const uint32_t goff = static_cast<uint32_t>(g) * kGroupPitch;
    if (rows == C::R && slot0 + C::R <= static_cast<size_t>(a.capacity)) {
      bulk_g2s(stage_dst + goff, src + slot0 * kRowBytes, C::R * kRowBytes, fb);
    } else {  // a partial group, or one that wraps around the ring: row by row
      for (int r = 0; r < rows; ++r) {
        const size_t slot = static_cast<size_t>((pos0 + r) % a.capacity);
        bulk_g2s(stage_dst + goff + r * kRowBytes, src + slot * kRowBytes, kRowBytes, fb);
      }
    }
  }
}

// Atomic increment with wrap ((old >= limit) ? 0 : old + 1) and
// acquire-release semantics at GPU scope; returns the old value.
__device__ __forceinline__ unsigned atom_inc_acq_rel(unsigned* p, unsigned limit) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.inc.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(limit) : "memory");
  return old;
}

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}


// A producer warp's last step: wait (bounded, with its own failure flag) for
// the last phase it issued into each stage of the ring, so no copy of this
// block is still in flight when the block exits. Earlier phases of a stage
// completed before that stage was issued again, and only the producers
// arrive on the full barriers, so the last issued phase is the last phase.
template <class C>
__device__ __forceinline__ void producer_drain(uint32_t full0, uint32_t st_issued, uint32_t st_par) {
  bool dfail = false;
#pragma unroll
  for (int st = 0; st < C::NSTAGE; ++st)
    if ((st_issued >> st) & 1u) mbar_wait(full0 + 8 * st, (st_par >> st) & 1u, dfail);
}

constexpr int kFusedLast = 1;   // fd_plan_t.fused values
constexpr int kFusedGroup = 2;

// The split kernel's body. PERSIST: the persistent grid; FUSED: the merge in
// the split launch (kFusedLast: the last block of each group merges;
// kFusedGroup: every block of a group waits for the group, then merges a
// share of its outputs). Each is a separate instance, so the plain per-split
// kernel keeps its registers (on GB300 every register it gains can keep the
// merge kernel's blocks, which wait beside it under programmatic dependent
// launch, off the SM).
template <class C, bool PERSIST, int FUSED>
__device__ __forceinline__ void split_tc_body(const LaunchArgs& a) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int s_seq[kLptMaxB];
  __shared__ int s_item[kItemQ];
  __shared__ __align__(8) uint64_t s_ibar[2 * kItemQ];  // work item queue: full[], empty[]
  const int G = a.NH / a.NKV;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  float* sS = reinterpret_cast<float*>(smem + C::OFF_S);
  uint16_t* sP = reinterpret_cast<uint16_t*>(smem + C::OFF_P);
  float* sAlpha = reinterpret_cast<float*>(smem + C::OFF_A);
  float* sM = sAlpha + C::NP;
  float* sL = sM + C::NP;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + C::NSTAGE);

  // Set-up that reads no input, overlapping the previous kernel's tail.
  if (tid == 0) {
    for (int i = 0; i < C::NSTAGE; ++i) {
      mbar_init(full0 + 8 * i, 64);         // every lane of both producer warps arrives once per phase
      mbar_init(empty0 + 8 * i, C::NWC);    // one arrival per consumer warp
    }
    for (int i = 0; i < kItemQ; ++i) {
      mbar_init(smem_u32(s_ibar + i), 1);                   // the K producer publishes
      mbar_init(smem_u32(s_ibar + kItemQ + i), C::NWC + 1);  // consumer warps and the V producer took it
    }
    fence_mbar_init();
  }
  // Start P at zero and alpha at 1 so nothing read before its first write can
  // carry a NaN bit pattern from uninitialised shared memory.
  for (int i = tid; i < 2 * C::NP * C::PPITCH; i += C::THREADS) sP[i] = 0;
  for (int i = tid; i < C::NP; i += C::THREADS) {
    sAlpha[i] = 1.f;
    sM[i] = kNegInf;
    sL[i] = 0.f;
  }
  // With no window, or a window as long as the cache, a band's slots are
  // [0, band), and the splits take its T-position tiles in turn (split s:
  // tiles s, s + S, s + 2S, ...), so a split's tiles are known before the
  // length is, and the tiles of slots [0, min(min_len, capacity)) are live
  // for every length the caller allows (min_len, the plan's lower bound). A
  // per-split block whose sequence needs no ordering table asks L2 for its
  // first such tile while the previous kernel is still running (a hint only:
  // nothing is read into the block before the dependency wait) and, past the
  // wait, copies it into stage 0 at once, before its length arrives. Nothing
  // else is read before the length is known, so only live slots are read.
  // (If a length breaks the bound, a tile copied early that the band does not
  // reach is never used: the producers wait for its copies before leaving.)
  // Measured on GB300 (us per layer; ring / MQA 32k / MQA 4k / Llama tiny):
  // the first tile requested and copied early 6.14 / 19.7 / 8.88 / 5.08;
  // the first NSTAGE tiles copied early 6.20 / 19.7 / 9.00 / 5.00; every sure
  // tile requested from L2 (up to a quarter of L2 over the grid) 6.20 / 21.7
  // / 9.00 / 5.08 (the requests delay the first tile's copies); nothing
  // requested, the first tiles copied early 6.66 / 20.1 / 9.06 / 5.25.
  constexpr int kRowBytesT = C::KV8 ? C::ROWB8 : C::ROWB;
  constexpr int kTileBytes = C::T * kRowBytesT;  // one tensor's bytes of one tile
  const bool tiled = a.window <= 0 || a.window >= a.capacity;
  const bool len_early = !PERSIST && !lpt_ordered(a);
  int n_sure = 0;  // this split's tiles that every allowed length makes live
  if (len_early && tiled) {
    const int nt_sure = min(a.min_len, a.capacity) / C::T;
    const int s0 = static_cast<int>(blockIdx.x);
    n_sure = nt_sure > s0 ? (nt_sure - s0 + a.num_splits - 1) / a.num_splits : 0;
  }
  const int n_early = min(min(n_sure, 1), max(0, a.withhold_tile));  // copied before the length is read
  if (n_sure > 0 && warp >= C::NWC && lane == 0)
    prefetch_l2(producer_src<C>(a, warp == C::NWC, blockIdx.z, blockIdx.y) +
                    static_cast<long long>(blockIdx.x) * kTileBytes, kTileBytes);
  // The block's query rows (G consecutive heads, contiguous) do not depend on
  // the length: ask L2 for them too.
  if (len_early && tid == 0)
    prefetch_l2(a.q + (static_cast<size_t>(blockIdx.z) * a.NH + static_cast<size_t>(blockIdx.y) * G) * C::HS,
                static_cast<uint32_t>(G) * C::HS * 2);
  grid_dependency_wait();
  grid_launch_dependents();
  // Such a block also reads its length before the barrier, so the load's
  // latency overlaps the barrier wait.
  const int len_first = len_early ? a.lens[blockIdx.z] : 0;
  lpt_table(a, tid, C::THREADS, s_seq);
  __syncthreads();

  // Stage-ring bookkeeping of a producer warp: the stages it has issued copies
  // into, and the phase parity of each stage's last issue (for the drain).
  uint32_t st_issued = 0, st_par = 0;
  if (n_early > 0 && warp >= C::NWC) {
    const bool is_k = warp == C::NWC;
    const unsigned char* src = producer_src<C>(a, is_k, blockIdx.z, blockIdx.y);
    constexpr size_t kStageBytes = C::KV8 ? C::STAGE8_BYTES : C::STAGE_BYTES;
    const uint32_t ring = smem_u32(smem + producer_ring<C>(is_k));
    for (int i = 0; i < n_early; ++i) {  // tiles 0 .. n_early - 1 of the split: stages 0 .. n_early - 1
      produce_tile<C>(a, src, ring + static_cast<uint32_t>(i * kStageBytes), full0 + 8 * i,
                      (static_cast<long long>(blockIdx.x) + static_cast<long long>(i) * a.num_splits) * C::T, C::T,
                      lane);
      st_issued |= 1u << i;
    }
  }

  // One work item (sequence, KV head, split) per block, or with a persistent
  // grid a stream of them: the K producer's lane 0 takes the next item index
  // from the counter and publishes it in a small shared-memory queue; the V
  // producer and the consumers read it from there. The counter wraps to zero
  // as the last block takes its final (past-the-end) index, so it is zero
  // again for the next call. Producers run ahead into the next item while the
  // consumers finish the current one: the stage ring and its phases continue
  // across items (gbase counts the tiles of earlier items).
  constexpr bool persist = PERSIST;  // a separate instantiation: the per-split grid keeps its registers
  const int n_items = persist ? a.num_splits * a.NKV * a.B : 1;
  bool failed = false;
  int gnext = 0;
  for (int it = 0;; ++it) {
  int s, kvh, z;
  if (!persist) {
    if (it > 0) break;
    s = blockIdx.x;
    kvh = blockIdx.y;
    z = blockIdx.z;
  } else {
    const int qi = it % kItemQ;
    const uint32_t ifull = smem_u32(s_ibar + qi), iempty = smem_u32(s_ibar + kItemQ + qi);
    int w = 0;
    if (warp == C::NWC) {
      if (lane == 0) {
        // take an index even after a failed wait, so the counter still wraps
        if (it >= kItemQ) mbar_wait(iempty, ((it / kItemQ) - 1) & 1, failed);
        w = static_cast<int>(atomicInc(a.work_counter, static_cast<unsigned>(n_items + gridDim.x - 1)));
        s_item[qi] = w;
        mbar_arrive(ifull);
      }
      w = __shfl_sync(0xffffffffu, w, 0);
    } else {
      w = mbar_wait(ifull, (it / kItemQ) & 1, failed) ? s_item[qi] : n_items;
      __syncwarp();
      if (lane == 0) mbar_arrive(iempty);
    }
    if (w >= n_items) break;
    s = w % a.num_splits;
    kvh = (w / a.num_splits) % a.NKV;
    z = w / (a.num_splits * a.NKV);
  }
  const int b = lpt_ordered(a) ? s_seq[z] : z;
  const int hbase = kvh * G;

  int lo;
  const int len_b = len_early ? len_first : a.lens[b];
  const bool reporter = s == 0 && kvh == 0 && tid == 0;
  if (reporter && len_b < a.min_len) atomicOr(&g_device_error, FD_DEVERR_MIN_LEN);
  const int band = band_of(len_b, a.capacity, a.window, reporter, &lo);
  // This split's tiles: tile i holds positions [tile_pos(i), + tile_nv(i)).
  // Tiled bands (slots [0, band)): tiles s, s + S, ... of the band; other
  // bands: the consecutive positions [lo + s*chunk, ...) cut into tiles. The
  // softmax does not depend on the order.
  const int S = a.num_splits;
  const int nt_band = (band + C::T - 1) / C::T;
  const int chunk = chunk_of(band, S, a.granule);
  const long long p0 = lo + static_cast<long long>(s) * chunk;
  const int n = tiled ? 0 : static_cast<int>(max(0ll, min(static_cast<long long>(lo) + band, p0 + chunk) - p0));
  const int ntiles = tiled ? (s < nt_band ? (nt_band - s + S - 1) / S : 0) : (n + C::T - 1) / C::T;
  const int nact = tiled ? min(S, nt_band) : active_splits(band, chunk);  // splits with work
  auto tile_pos = [&](int i) -> long long {
    return tiled ? static_cast<long long>(s + i * S) * C::T : p0 + static_cast<long long>(i) * C::T;
  };
  auto tile_nv = [&](int i) -> int {
    return tiled ? min(C::T, band - (s + i * S) * C::T) : min(C::T, n - i * C::T);
  };
  const int CS = a.cluster;                 // blocks per cluster along the splits
  const bool direct = S == CS;              // one block / cluster spans every split

  if (ntiles == 0 && CS == 1) {
    // no copy may land after the block has left (tiles copied early for a
    // length below the plan's bound)
    if (!persist && warp >= C::NWC) producer_drain<C>(full0, st_issued, st_par);
    // len == 0: the output row is zero. With one block per band, or with an
    // in-launch merge (no block of an empty band ever merges), block 0 writes it.
    if (direct || (FUSED && band == 0 && s == 0)) {
      for (int i = tid; i < G * C::HS; i += C::THREADS) {
        const size_t o = (static_cast<size_t>(b) * a.NH + hbase + i / C::HS) * C::HS + i % C::HS;
        a.out[o] = 0;
        if (a.out_f32) a.out_f32[o] = 0.f;
      }
    } else if (!FUSED) {
      write_empty_partial(a, b, hbase, G, C::HS, s, tid, C::THREADS);
    }
    continue;
  }
  // In a cluster every block, even one with an empty slice (m = -inf, l = 0,
  // O = 0), takes part in the reduction at the end.
  const int gbase = gnext;  // pipeline tiles of this block's earlier items
  gnext = gbase + ntiles;

  const int grp = lane >> 2, t4 = lane & 3;
  const int dbase = warp * C::DW;
  float o[C::KD][C::NT][4];
#pragma unroll
  for (int mt = 0; mt < C::KD; ++mt)
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.f;
  // softmax role: row sr, MMA rows sj + tpr * t; when the real query rows
  // fit half of the padded ones, only those are taken, with twice the
  // threads per row (the padded rows' P stays 0, their alpha 1, and they feed
  // only accumulator columns that are never stored)
  const bool half_rows = C::TPR2 > C::TPR && 2 * G <= C::NP;
  const int tpr_rt = half_rows ? C::TPR2 : C::TPR;
  const int sr = tid / tpr_rt, sj = tid % tpr_rt;

  if (warp >= C::NWC) {
    // ----------------------------------------------------------- producers
    // Warp NWC streams K, warp NWC + 1 streams V: two issuing warps raise a
    // block's copy rate (a block's rate is set by the copies it issues).
    const bool is_k = warp == C::NWC;
    const unsigned char* src = producer_src<C>(a, is_k, b, kvh);
    constexpr size_t kStageBytes = C::KV8 ? C::STAGE8_BYTES : C::STAGE_BYTES;
    const size_t ring = producer_ring<C>(is_k);
    for (int i = persist ? 0 : n_early; i < ntiles; ++i) {  // tiles [0, n_early) are in flight already
      if (!persist && i >= a.withhold_tile) break;              // test hook: these copies are never issued
      const int gi = gbase + i;
      const int st = gi % C::NSTAGE;
      if (gi >= C::NSTAGE) mbar_wait(empty0 + 8 * st, ((gi / C::NSTAGE) - 1) & 1, failed);
      if (persist && failed) continue;  // nothing waits for these copies any more
      const int nv = tile_nv(i);
      const long long pbase = tile_pos(i);
      produce_tile<C>(a, src, smem_u32(smem + ring + static_cast<size_t>(st) * kStageBytes), full0 + 8 * st, pbase,
                      nv, lane);
      st_issued |= 1u << st;
      st_par = (st_par & ~(1u << st)) | (static_cast<uint32_t>((gi / C::NSTAGE) & 1) << st);
    }
    // Every copy this warp issued has landed before the block can leave: a
    // consumer wait that gave up must not leave copies in flight.
    if (!persist) producer_drain<C>(full0, st_issued, st_par);
  } else {
  // -------------------------------------------------------------- consumers

  // Q^T as MMA B fragments for this warp's dims: b0 = (dims 2t4..2t4+1, row grp),
  // b1 = (dims 8+2t4.., row grp) of each 16-dim step; for KV8 (k slots =
  // consecutive dims) b0 = dims 4t4..4t4+1, b1 = dims 4t4+2..4t4+3.
  constexpr int kQLo = C::KV8 ? 4 : 2, kQHi = C::KV8 ? 2 : 8;
  uint32_t qf[C::KD][C::NT][2];
#pragma unroll
  for (int ks = 0; ks < C::KD; ++ks)
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt) {
      const int r = nt * 8 + grp;
      uint32_t x0 = 0, x1 = 0;
      if (r < G) {
        const uint16_t* qr = a.q + (static_cast<size_t>(b) * a.NH + hbase + r) * C::HS + dbase + ks * 16 + kQLo * t4;
        x0 = *reinterpret_cast<const uint32_t*>(qr);
        x1 = *reinterpret_cast<const uint32_t*>(qr + kQHi);
      }
      qf[ks][nt][0] = x0;
      qf[ks][nt][1] = x1;
    }

  float sl2 = a.scale_log2;  // score scale, log2 units
  // E4M3: this head's K and V scales, loaded now so their latency is not on
  // the path to the first scores or to the epilogue
  [[maybe_unused]] float k_scale = 1.f, v_scale = 1.f;
  if constexpr (C::KV8) {
    k_scale = a.k_scale[static_cast<size_t>(b) * a.NKV + kvh];
    v_scale = a.v_scale[static_cast<size_t>(b) * a.NKV + kvh];
  }
  if constexpr (C::KV8) {
    // fp16 MMAs: Q goes to fp16 with one power-of-two scale per block, so the
    // block's largest |q| lands in [2^13, 2^14) and no product can overflow;
    // that scale and the K dequantisation scale fold into the score scale.
    __shared__ float s_qmax[C::NWC];
    float qmax = 0.f;
#pragma unroll
    for (int ks = 0; ks < C::KD; ++ks)
#pragma unroll
      for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const uint32_t x = qf[ks][nt][e];
          qmax = fmaxf(qmax, fmaxf(fabsf(bf16_bits_to_f32(static_cast<uint16_t>(x & 0xffffu))),
                                   fabsf(bf16_bits_to_f32(static_cast<uint16_t>(x >> 16)))));
        }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, off));
    if (lane == 0) s_qmax[warp] = qmax;
    named_bar_sync(1, C::CTHREADS);
#pragma unroll
    for (int w = 0; w < C::NWC; ++w) qmax = fmaxf(qmax, s_qmax[w]);
    const int eq = (qmax > 0.f && qmax <= 3.0e38f) ? 13 - ilogbf(qmax) : 0;
#pragma unroll
    for (int ks = 0; ks < C::KD; ++ks)
#pragma unroll
      for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const uint32_t x = qf[ks][nt][e];
          qf[ks][nt][e] = pack_f16x2(ldexpf(bf16_bits_to_f32(static_cast<uint16_t>(x & 0xffffu)), eq),
                                     ldexpf(bf16_bits_to_f32(static_cast<uint16_t>(x >> 16)), eq));
        }
    sl2 = a.scale_log2 * k_scale * ldexpf(1.f, -eq);
  }

  float m_run = kNegInf, l_run = 0.f;

  // ldmatrix lane addressing
  const int lrow = lane & 7, lmat = lane >> 3;

  for (int i = 0; i < ntiles; ++i) {
    const int gi = gbase + i;
    const int st = gi % C::NSTAGE;
    mbar_wait(full0 + 8 * st, (gi / C::NSTAGE) & 1, failed);
    const int nv = tile_nv(i);  // valid tile positions: [0, nv)
    const unsigned char* tK = smem + C::OFF_K + static_cast<size_t>(st) * C::STAGE_BYTES;
    unsigned char* tV = smem + C::OFF_V + static_cast<size_t>(st) * C::STAGE_BYTES;
    // E4M3 stage (KV8)
    [[maybe_unused]] const unsigned char* fK = smem + C::OFF_K8 + static_cast<size_t>(st) * C::STAGE8_BYTES;
    [[maybe_unused]] const unsigned char* fV = smem + C::OFF_V8 + static_cast<size_t>(st) * C::STAGE8_BYTES;

    // ---- scores: S^T[m][row] partial over this warp's dims (m = MMA row order)
    float* myS = sS + static_cast<size_t>(warp) * C::NP * C::SP;
#pragma unroll
    for (int mt = 0; mt < C::MP; ++mt) {
      if (C::min_pos(mt) < nv) {
        float acc[C::NT][4];
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[nt][e] = 0.f;
        if constexpr (C::KV8) {
          // rows mt*16 + grp and + 8; k slots 2t4, 2t4+1 / 2t4+8, 2t4+9 = dims 4t4 .. 4t4+3
          const unsigned char* k0 = fK + C::off8_of(mt * 16 + grp) + dbase + 4 * t4;
#pragma unroll
          for (int ks = 0; ks < C::KD; ++ks) {
            const uint32_t w0 = *reinterpret_cast<const uint32_t*>(k0 + ks * 16);
            const uint32_t w1 = *reinterpret_cast<const uint32_t*>(k0 + C::ROWB8 + ks * 16);
            const uint32_t a0 = e4m3x2_to_f16x2(static_cast<uint16_t>(w0 & 0xffffu));
            const uint32_t a2 = e4m3x2_to_f16x2(static_cast<uint16_t>(w0 >> 16));
            const uint32_t a1 = e4m3x2_to_f16x2(static_cast<uint16_t>(w1 & 0xffffu));
            const uint32_t a3 = e4m3x2_to_f16x2(static_cast<uint16_t>(w1 >> 16));
#pragma unroll
            for (int nt = 0; nt < C::NT; ++nt)
              mma_f16_16816(acc[nt], a0, a1, a2, a3, qf[ks][nt][0], qf[ks][nt][1]);
          }
        } else {
#pragma unroll
          for (int ks = 0; ks < C::KD; ++ks) {
            // matrices: (rows 0-7, d 0-7), (rows 8-15, d 0-7), (rows 0-7, d 8-15), (rows 8-15, d 8-15)
            const int m = mt * 16 + lrow + (lmat & 1) * 8;
            const int dcol = dbase + ks * 16 + (lmat >> 1) * 8;
            uint32_t a0, a1, a2, a3;
            ldsm_x4(smem_u32(tK + C::off_of(m) + dcol * 2), a0, a1, a2, a3);
#pragma unroll
            for (int nt = 0; nt < C::NT; ++nt)
              mma_bf16_16816(acc[nt], a0, a1, a2, a3, qf[ks][nt][0], qf[ks][nt][1]);
          }
        }
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt) {
          float* d0 = myS + (nt * 8 + 2 * t4) * C::SP + mt * 16 + grp;  // [row][MMA row]
          d0[0] = acc[nt][0];
          d0[C::SP] = acc[nt][1];
          d0[8] = acc[nt][2];
          d0[C::SP + 8] = acc[nt][3];
        }
      }
    }
    named_bar_sync(1, C::CTHREADS);

    // ---- one online-softmax update per row for the whole tile. Every
    // consumer thread takes part (padded rows >= G included unless the half
    // mapping leaves them out), so the full-warp shuffles below never run in a
    // partial warp; padded rows only feed accumulator columns that are never
    // stored.
    auto softmax_rows = [&](auto tpr_c) {
      constexpr int TPRx = decltype(tpr_c)::value;
      constexpr int PPTx = C::T / TPRx;
      float sv[PPTx];
      float tmax = kNegInf;
#pragma unroll
      for (int t = 0; t < PPTx; ++t) {
        const int j = sj + t * TPRx;  // MMA row
        float x = kNegInf;
        if (C::pos_of(j) < nv) {
          float acc = 0.f;
#pragma unroll
          for (int w = 0; w < C::NWC; ++w) acc += sS[(static_cast<size_t>(w) * C::NP + sr) * C::SP + j];
          x = acc * sl2;
        }
        sv[t] = x;
        tmax = fmaxf(tmax, x);
        if (isnan(x)) tmax = x;
      }
#pragma unroll
      for (int off = TPRx / 2; off > 0; off >>= 1) {
        const float other = __shfl_xor_sync(0xffffffffu, tmax, off);
        tmax = isnan(other) ? other : fmaxf(tmax, other);
      }
      const float m_new = isnan(tmax) ? tmax : fmaxf(m_run, tmax);
      const float alpha = (m_new == kNegInf) ? 1.f : exp2f(m_run - m_new);
      float psum = 0.f;
      uint16_t* phi = sP + sr * C::PPITCH;
      [[maybe_unused]] uint16_t* plo = sP + (C::NP + sr) * C::PPITCH;  // bf16 tiles: the low halves of P
#pragma unroll
      for (int t = 0; t < PPTx; ++t) {
        const int j = sj + t * TPRx;
        const float p = exp2f(sv[t] - m_new);
        if constexpr (C::KV8) {
          phi[j] = __half_as_ushort(__float2half_rn(p));  // fp16 P: 11 bits, no second pass
        } else {
          const uint16_t hi = f32_to_bf16_bits(p);
          const uint16_t lo16 = f32_to_bf16_bits(p - bf16_bits_to_f32(hi));
          phi[j] = hi;
          plo[j] = lo16;
        }
        psum += p;
      }
#pragma unroll
      for (int off = TPRx / 2; off > 0; off >>= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
      l_run = l_run * alpha + psum;
      m_run = m_new;
      if (sj == 0) sAlpha[sr] = alpha;
    };
    if constexpr (C::TPR2 > C::TPR) {
      if (half_rows) {
        softmax_rows(std::integral_constant<int, C::TPR2>{});
      } else {
        softmax_rows(std::integral_constant<int, C::TPR>{});
      }
    } else {
      softmax_rows(std::integral_constant<int, C::TPR>{});
    }
    // V rows of positions [nv, T) were not written by this tile's copies:
    // zero them so 0-weight positions contribute exactly 0.
    if (!C::KV8 && nv < C::T) {
      const int words = (C::T - nv) * (C::HS / 8);  // 16-byte words
      for (int w16 = tid; w16 < words; w16 += C::CTHREADS) {
        const int r = nv + w16 / (C::HS / 8), c = (w16 % (C::HS / 8)) * 16;
        *reinterpret_cast<uint4*>(tV + C::off_pos(r) + c) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();  // order before the next bulk copies into this stage
    }
    named_bar_sync(1, C::CTHREADS);

    // ---- O^T[dim][row] = alpha * O^T + V^T P^T  (P split into bf16 hi + lo; one fp16 P for KV8)
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt) {
      const float al0 = sAlpha[nt * 8 + 2 * t4], al1 = sAlpha[nt * 8 + 2 * t4 + 1];
      // once the running maxima settle, alpha is exactly 1 for every row: skip
      // the multiplies (x * 1 == x, so the result is the same either way)
      if (!__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) continue;
#pragma unroll
      for (int mt = 0; mt < C::KD; ++mt) {
        o[mt][nt][0] *= al0;
        o[mt][nt][1] *= al1;
        o[mt][nt][2] *= al0;
        o[mt][nt][3] *= al1;
      }
    }
#pragma unroll
    for (int kp = 0; kp < C::MP; ++kp) {
      if (C::min_pos(kp) < nv) {
        uint32_t pb[C::NT][4];
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt) {
          // matrices: (hi, pos 0-7), (hi, pos 8-15), (lo, pos 0-7), (lo, pos 8-15); rows = query rows
          const uint16_t* pa = sP + ((lmat >> 1) * C::NP + nt * 8 + lrow) * C::PPITCH + kp * 16 + (lmat & 1) * 8;
          if constexpr (C::KV8) {
            ldsm_x2(smem_u32(pa), pb[nt][0], pb[nt][1]);  // fp16 P: no lo half
          } else {
            ldsm_x4(smem_u32(pa), pb[nt][0], pb[nt][1], pb[nt][2], pb[nt][3]);
          }
        }
        if constexpr (C::KV8) {
          // k slots 2t4, 2t4+1, 2t4+8, 2t4+9 are MMA rows m0, m0+1, m0+8, m0+9;
          // a load of a row past the tile's valid positions reads 0 instead
          // (its P is 0, and stale codes may be NaN).
          const int m0 = kp * 16 + 2 * t4;
          const int mr[4] = {m0, m0 + 1, m0 + 8, m0 + 9};
          const unsigned char* vr[4];
          bool ok[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            vr[i] = fV + C::off8_of(mr[i]) + dbase + 4 * grp;
            ok[i] = C::pos_of(mr[i]) < nv;
          }
#pragma unroll
          for (int c = 0; c < C::DW / 32; ++c) {
            uint32_t L[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) L[i] = ok[i] ? *reinterpret_cast<const uint32_t*>(vr[i] + 32 * c) : 0u;
            // byte j of L[i] = dim 4 grp + j of row mr[i]; pair rows (0,1) and (2,3) per dim
            const uint32_t x01 = __byte_perm(L[0], L[1], 0x5140), x23 = __byte_perm(L[2], L[3], 0x5140);
            const uint32_t y01 = __byte_perm(L[0], L[1], 0x7362), y23 = __byte_perm(L[2], L[3], 0x7362);
            const uint32_t a0 = e4m3x2_to_f16x2(static_cast<uint16_t>(x01 & 0xffffu));  // dim +0
            const uint32_t a1 = e4m3x2_to_f16x2(static_cast<uint16_t>(x01 >> 16));      // dim +1
            const uint32_t a2 = e4m3x2_to_f16x2(static_cast<uint16_t>(x23 & 0xffffu));
            const uint32_t a3 = e4m3x2_to_f16x2(static_cast<uint16_t>(x23 >> 16));
            const uint32_t b0 = e4m3x2_to_f16x2(static_cast<uint16_t>(y01 & 0xffffu));  // dim +2
            const uint32_t b1 = e4m3x2_to_f16x2(static_cast<uint16_t>(y01 >> 16));      // dim +3
            const uint32_t b2 = e4m3x2_to_f16x2(static_cast<uint16_t>(y23 & 0xffffu));
            const uint32_t b3 = e4m3x2_to_f16x2(static_cast<uint16_t>(y23 >> 16));
#pragma unroll
            for (int nt = 0; nt < C::NT; ++nt) {
              mma_f16_16816(o[2 * c][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
              mma_f16_16816(o[2 * c + 1][nt], b0, b1, b2, b3, pb[nt][0], pb[nt][1]);
            }
          }
        } else {
#pragma unroll
          for (int mt = 0; mt < C::KD; ++mt) {
            // V^T fragments: matrices (d 0-7, rows 0-7), (d 8-15, rows 0-7), (d 0-7, rows 8-15), (d 8-15, rows 8-15)
            const int m = kp * 16 + lrow + (lmat >> 1) * 8;
            const int dcol = dbase + mt * 16 + (lmat & 1) * 8;
            uint32_t v0, v1, v2, v3;
            ldsm_x4_trans(smem_u32(tV + C::off_of(m) + dcol * 2), v0, v1, v2, v3);
#pragma unroll
            for (int nt = 0; nt < C::NT; ++nt) {
              mma_bf16_16816(o[mt][nt], v0, v1, v2, v3, pb[nt][0], pb[nt][1]);
              mma_bf16_16816(o[mt][nt], v0, v1, v2, v3, pb[nt][2], pb[nt][3]);
            }
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * st);
  }

    if constexpr (C::KV8) {  // O in dequantised units: times this head's V scale
      const float vs = v_scale;
#pragma unroll
      for (int mt = 0; mt < C::KD; ++mt)
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) o[mt][nt][e] *= vs;
    }
    if (sr < G && sj == 0) {
      sM[sr] = m_run;
      sL[sr] = l_run;
    }
    named_bar_sync(1, C::CTHREADS);  // every consumer is past its last tile
  }

  if (CS == 1) {
    // ---- one block per slice: its partial (O, m, l), or with one split the
    // normalised row
    if (warp >= C::NWC) continue;
#pragma unroll
    for (int mt = 0; mt < C::KD; ++mt)
#pragma unroll
      for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = nt * 8 + 2 * t4 + (e & 1);
          if (r >= G) continue;
          const int d = dbase + C::dim_of(mt, grp, e >> 1);
          const size_t row = static_cast<size_t>(b) * a.NH + hbase + r;
          if (direct) {
            const float val = o[mt][nt][e] / sL[r];
            a.out[row * C::HS + d] = f32_to_bf16_bits(val);
            if (a.out_f32) a.out_f32[row * C::HS + d] = val;
          } else {
            a.ws_o[(row * a.num_splits + s) * C::HS + d] = o[mt][nt][e];
          }
        }
    if (!direct && tid < G) {
      const size_t r = ((static_cast<size_t>(b) * a.NH + hbase + tid) * a.num_splits + s) * 2;
      a.ws_ml[r] = sM[tid];
      a.ws_ml[r + 1] = sL[tid];
    }
    if constexpr (!FUSED) continue;
    if (direct) continue;

    if constexpr (FUSED == kFusedGroup) {
      // ---- group step: every active block of this (sequence, KV head) counts
      // in, waits until the whole group has, then merges its share of the
      // group's G x HS outputs. The grid is launched cooperatively (every
      // block resident at once), so the wait ends; it is bounded all the
      // same. Thread 0 counts the block in with an acquire-release add (the
      // barrier before it orders the block's partial stores first), so the
      // last arrival has observed every partial, and waits with acquire loads
      // until the count is complete, which passes that view on (and, through
      // the barrier after the wait, to the block). Each block then counts out
      // on a second word; the last one out sets both words back to zero for
      // the next call (every other block has seen the full count by then).
      __shared__ int s_go;
      unsigned* cnt = a.counters + static_cast<size_t>(b) * a.NKV + kvh;
      unsigned* out_cnt = cnt + static_cast<size_t>(a.B) * a.NKV;
      named_bar_sync(1, C::CTHREADS);
      if (tid == 0) {
        int go = 1;
        const unsigned need = static_cast<unsigned>(nact);
        if (atom_add_acq_rel(cnt, 1u) + 1u < need) {
          uint64_t t0 = 0;
          for (uint32_t i = 1; ld_acquire_u32(cnt) < need; ++i) {
            if ((i & 255u) != 0) continue;  // the clock is read every 256 polls
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) {
              t0 = now;
            } else if (now - t0 > g_wait_limit_ns) {
              go = 0;
              atomicOr(&g_device_error, FD_DEVERR_WAIT_TIMEOUT);
              break;
            }
          }
        }
        if (go && atomicAdd(out_cnt, 1u) == need - 1u) {
          *reinterpret_cast<volatile unsigned*>(cnt) = 0u;
          *reinterpret_cast<volatile unsigned*>(out_cnt) = 0u;
        }
        s_go = go;
      }
      named_bar_sync(1, C::CTHREADS);
      if (!s_go) return;

      // Block s of the nact active ones takes items [s * per, (s + 1) * per)
      // of the group's (row, 4 dims) items. A warp takes 32 / LG items at
      // once, LG lanes each (the power of two >= nact, at most 32); the lanes
      // of an item take its slots sl, sl + LG, ... with every load in flight
      // at once, fold them online, and combine with a butterfly inside the
      // LG lanes, which gives each of them the same, order-fixed sum.
      const int S = a.num_splits;
      constexpr int D4 = C::HS / 4;
      constexpr int kLoads = 8;  // slots per lane per round trip
      const int items = G * D4;
      const int per = (items + nact - 1) / nact;
      const int i_end = min(items, (s + 1) * per);
      int LG = 1;
      while (LG < nact && LG < 32) LG <<= 1;
      const int ipw = 32 / LG, sub = lane / LG, sl = lane % LG;
      for (int it0 = s * per + warp * ipw; it0 < i_end; it0 += C::NWC * ipw) {
        const int it = min(it0 + sub, i_end - 1);  // lanes past the end repeat the last item, unstored
        const int g = it / D4, d = (it % D4) * 4;
        const size_t row = static_cast<size_t>(b) * a.NH + hbase + g;
        const float4* src = reinterpret_cast<const float4*>(a.ws_o + row * S * C::HS + d);
        const float2* ml = reinterpret_cast<const float2*>(a.ws_ml) + row * S;
        float M = kNegInf, L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j0 = sl; j0 < nact; j0 += LG * kLoads) {
          float4 v[kLoads];
          float2 w2[kLoads];
#pragma unroll
          for (int u = 0; u < kLoads; ++u) {
            const int j = j0 + LG * u;
            v[u] = j < nact ? __ldcg(src + static_cast<size_t>(j) * D4) : make_float4(0.f, 0.f, 0.f, 0.f);
            w2[u] = j < nact ? __ldcg(ml + j) : make_float2(kNegInf, 0.f);
          }
          float bm = kNegInf;
#pragma unroll
          for (int u = 0; u < kLoads; ++u) bm = fmaxf(bm, w2[u].x);
          const float mn = fmaxf(M, bm);
          if (mn == kNegInf) continue;
          const float sc = exp2f(M - mn);  // 0 while M is still -inf
          L *= sc;
          acc.x *= sc;
          acc.y *= sc;
          acc.z *= sc;
          acc.w *= sc;
#pragma unroll
          for (int u = 0; u < kLoads; ++u) {
            const float w = exp2f(w2[u].x - mn);  // 0 for padding and empty partials; NaN for a NaN m
            L += w * w2[u].y;
            acc.x += w * v[u].x;
            acc.y += w * v[u].y;
            acc.z += w * v[u].z;
            acc.w += w * v[u].w;
          }
          M = mn;
        }
        for (int off = LG >> 1; off > 0; off >>= 1) {
          const float Mo = __shfl_xor_sync(0xffffffffu, M, off);
          const float Lo = __shfl_xor_sync(0xffffffffu, L, off);
          const float4 ao = make_float4(__shfl_xor_sync(0xffffffffu, acc.x, off),
                                        __shfl_xor_sync(0xffffffffu, acc.y, off),
                                        __shfl_xor_sync(0xffffffffu, acc.z, off),
                                        __shfl_xor_sync(0xffffffffu, acc.w, off));
          const float mn = fmaxf(M, Mo);
          const float sa = M == kNegInf ? 0.f : exp2f(M - mn);
          const float sb = Mo == kNegInf ? 0.f : exp2f(Mo - mn);
          L = L * sa + Lo * sb;
          acc.x = acc.x * sa + ao.x * sb;
          acc.y = acc.y * sa + ao.y * sb;
          acc.z = acc.z * sa + ao.z * sb;
          acc.w = acc.w * sa + ao.w * sb;
          M = mn;
        }
        if (sl == 0 && it0 + sub < i_end) {
          const float4 val = make_float4(acc.x / L, acc.y / L, acc.z / L, acc.w / L);
          const uint32_t lo2 = static_cast<uint32_t>(f32_to_bf16_bits(val.x)) |
                               (static_cast<uint32_t>(f32_to_bf16_bits(val.y)) << 16);
          const uint32_t hi2 = static_cast<uint32_t>(f32_to_bf16_bits(val.z)) |
                               (static_cast<uint32_t>(f32_to_bf16_bits(val.w)) << 16);
          *reinterpret_cast<uint2*>(a.out + row * C::HS + d) = make_uint2(lo2, hi2);
          if (a.out_f32) *reinterpret_cast<float4*>(a.out_f32 + row * C::HS + d) = val;
        }
      }
      return;
    }

    // ---- fused merge: the last block of this (sequence, KV head) to finish
    // combines every partial of the group (no merge launch). Thread 0 counts
    // the block in with one acquire-release atomic: its release publishes the
    // block's partial stores (the barrier ordered them before it), its
    // acquire makes every earlier block's partials visible here (the barrier
    // after it passes that on to the block). The counter wraps to zero as the
    // last block takes it, so it is zero again for the next call. The last
    // block loads each (row, 4 dims) item's partials and their (m, l) in one
    // round trip per batch and folds them online; when there are fewer items
    // than threads, JG threads share an item's splits and meet in shared
    // memory in a fixed order.
    __shared__ int s_last;
    const int nsplit = nact;
    named_bar_sync(1, C::CTHREADS);  // every thread's partial stores precede thread 0's release
    if (tid == 0)
      s_last = atom_inc_acq_rel(a.counters + static_cast<size_t>(b) * a.NKV + kvh, static_cast<unsigned>(nsplit - 1)) ==
               static_cast<unsigned>(nsplit - 1);
    named_bar_sync(1, C::CTHREADS);
    if (!s_last) return;

    const int S = a.num_splits;
    constexpr int D4 = C::HS / 4;
    constexpr int kFusedBatch = 8;
    const int items = G * D4;
    int JG = C::CTHREADS / items;
    if (JG < 1 || static_cast<size_t>(JG) * items * 24 > static_cast<size_t>(C::NWC) * C::NP * C::SP * 4) JG = 1;
    float4* sAcc = reinterpret_cast<float4*>(sS);                 // [JG][items] weighted O sums
    float2* sMl = reinterpret_cast<float2*>(sAcc + JG * items);  // [JG][items] (max, weighted l)
    auto store_out = [&](size_t row, int d, float4 acc, float L) {
      const float4 val = make_float4(acc.x / L, acc.y / L, acc.z / L, acc.w / L);
      const uint32_t lo2 = static_cast<uint32_t>(f32_to_bf16_bits(val.x)) |
                           (static_cast<uint32_t>(f32_to_bf16_bits(val.y)) << 16);
      const uint32_t hi2 = static_cast<uint32_t>(f32_to_bf16_bits(val.z)) |
                           (static_cast<uint32_t>(f32_to_bf16_bits(val.w)) << 16);
      *reinterpret_cast<uint2*>(a.out + row * C::HS + d) = make_uint2(lo2, hi2);
      if (a.out_f32) *reinterpret_cast<float4*>(a.out_f32 + row * C::HS + d) = val;
    };
    for (int t = tid; t < items * JG; t += C::CTHREADS) {
      const int item = t % items, jg = t / items;
      const int g = item / D4, d = (item % D4) * 4;
      const size_t row = static_cast<size_t>(b) * a.NH + hbase + g;
      const float4* src = reinterpret_cast<const float4*>(a.ws_o + row * S * C::HS + d);
      const float2* ml = reinterpret_cast<const float2*>(a.ws_ml) + row * S;
      float M = kNegInf, L = 0.f;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j0 = jg; j0 < nsplit; j0 += kFusedBatch * JG) {
        float4 v[kFusedBatch];
        float2 w2[kFusedBatch];
#pragma unroll
        for (int u = 0; u < kFusedBatch; ++u) {  // every load of the batch in flight at once
          const int j = j0 + u * JG;
          v[u] = j < nsplit ? __ldcg(src + static_cast<size_t>(j) * D4) : make_float4(0.f, 0.f, 0.f, 0.f);
          w2[u] = j < nsplit ? __ldcg(ml + j) : make_float2(kNegInf, 0.f);
        }
        float bm = kNegInf;
#pragma unroll
        for (int u = 0; u < kFusedBatch; ++u) bm = fmaxf(bm, w2[u].x);
        const float mn = fmaxf(M, bm);
        if (mn == kNegInf) continue;  // nothing but empty partials so far
        const float sc = exp2f(M - mn);  // 0 while M is still -inf
        L *= sc;
        acc.x *= sc;
        acc.y *= sc;
        acc.z *= sc;
        acc.w *= sc;
#pragma unroll
        for (int u = 0; u < kFusedBatch; ++u) {
          const float w = exp2f(w2[u].x - mn);  // 0 for padding and empty partials
          L += w * w2[u].y;
          acc.x += w * v[u].x;
          acc.y += w * v[u].y;
          acc.z += w * v[u].z;
          acc.w += w * v[u].w;
        }
        M = mn;
      }
      if (JG == 1) {
        store_out(row, d, acc, L);
      } else {
        sAcc[jg * items + item] = acc;
        sMl[jg * items + item] = make_float2(M, L);
      }
    }
    if (JG > 1) {
      named_bar_sync(1, C::CTHREADS);
      for (int item = tid; item < items; item += C::CTHREADS) {
        const int g = item / D4, d = (item % D4) * 4;
        const size_t row = static_cast<size_t>(b) * a.NH + hbase + g;
        float M = kNegInf;
        for (int jg = 0; jg < JG; ++jg) M = fmaxf(M, sMl[jg * items + item].x);
        float L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int jg = 0; jg < JG; ++jg) {  // fixed order: the result does not depend on timing
          const float2 ml = sMl[jg * items + item];
          const float w = ml.x == kNegInf ? 0.f : exp2f(ml.x - M);
          const float4 o2 = sAcc[jg * items + item];
          L += w * ml.y;
          acc.x += w * o2.x;
          acc.y += w * o2.y;
          acc.z += w * o2.z;
          acc.w += w * o2.w;
        }
        store_out(row, d, acc, L);
      }
    }
    return;
  }

  // ---- cluster reduction through distributed shared memory. Each block parks
  // its unnormalised O (rows < G, fp32 [G][HS]) in its now idle K stages; after
  // a cluster barrier, block `rank` combines head dims
  // [rank * HS / CS, (rank + 1) * HS / CS) of every row over the CS blocks:
  // M = max_c m_c, w_c = 2^(m_c - M), O = sum_c w_c O_c, L = sum_c w_c l_c.
  // A block whose slice turned out empty (a length below the plan's bound)
  // may still have its first tile's early copies in flight into stage 0: they
  // must land before O is parked over that stage. A block with tiles waited
  // for every copy it issued when it consumed them.
  if (n_early > 0 && ntiles == 0 && warp < C::NWC) mbar_wait(full0, 0, failed);
  float* sO = reinterpret_cast<float*>(smem + C::OFF_K);
  if (warp < C::NWC) {
#pragma unroll
    for (int mt = 0; mt < C::KD; ++mt)
#pragma unroll
      for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int r = nt * 8 + 2 * t4 + (e & 1);
          if (r < G) sO[r * C::HS + dbase + C::dim_of(mt, grp, e >> 1)] = o[mt][nt][e];
        }
  }
  cluster_sync_all();

  const uint32_t rank = cluster_ctarank();
  float* sW = sS;                 // [G][CS] weights
  float* sMt = sS + G * CS;       // [G] combined max
  float* sLt = sMt + G;           // [G] combined sum
  if (tid < G) {
    float M = kNegInf;
    for (int c = 0; c < CS; ++c) M = fmaxf(M, ld_dsmem(map_to_rank(smem_u32(sM + tid), c)));
    float L = 0.f;
    for (int c = 0; c < CS; ++c) {
      const float mc = ld_dsmem(map_to_rank(smem_u32(sM + tid), c));
      const float lc = ld_dsmem(map_to_rank(smem_u32(sL + tid), c));
      const float w = (M == kNegInf) ? 0.f : exp2f(mc - M);
      sW[tid * CS + c] = w;
      L += w * lc;
    }
    sMt[tid] = M;
    sLt[tid] = L;
  }
  __syncthreads();

  const int dc4 = C::HS / CS / 4;  // float4 columns per block
  const int q = s / CS;            // this cluster's partial slot
  const int nq = a.num_splits / CS;
  for (int it = tid; it < G * dc4; it += C::THREADS) {
    const int r = it / dc4;
    const int d = static_cast<int>(rank) * (C::HS / CS) + (it % dc4) * 4;
    const uint32_t src = smem_u32(sO + r * C::HS + d);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int c = 0; c < CS; ++c) {
      const float w = sW[r * CS + c];
      const float4 v = ld_dsmem4(map_to_rank(src, c));
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
    }
    const size_t row = static_cast<size_t>(b) * a.NH + hbase + r;
    if (direct) {
      const float L = sLt[r];
      const float inv = L > 0.f ? 1.f / L : 0.f;
      const float4 val = (L > 0.f || isnan(L)) ? make_float4(acc.x / L, acc.y / L, acc.z / L, acc.w / L)
                                               : make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
      const uint32_t lo2 = static_cast<uint32_t>(f32_to_bf16_bits(val.x)) |
                           (static_cast<uint32_t>(f32_to_bf16_bits(val.y)) << 16);
      const uint32_t hi2 = static_cast<uint32_t>(f32_to_bf16_bits(val.z)) |
                           (static_cast<uint32_t>(f32_to_bf16_bits(val.w)) << 16);
      *reinterpret_cast<uint2*>(a.out + row * C::HS + d) = make_uint2(lo2, hi2);
      if (a.out_f32) *reinterpret_cast<float4*>(a.out_f32 + row * C::HS + d) = val;
    } else {
      *reinterpret_cast<float4*>(a.ws_o + (row * nq + q) * C::HS + d) = acc;
    }
  }
  if (!direct && rank == 0 && tid < G) {
    const size_t r = ((static_cast<size_t>(b) * a.NH + hbase + tid) * nq + q) * 2;
    a.ws_ml[r] = sMt[tid];
    a.ws_ml[r + 1] = sLt[tid];
  }
  cluster_sync_all();  // no block leaves while another still reads its shared memory
  }  // work items
  if (PERSIST && warp >= C::NWC) producer_drain<C>(full0, st_issued, st_par);
}

template <class C, bool PERSIST = false, int FUSED = 0>
__global__ void __launch_bounds__(C::THREADS, FUSED ? C::MINB : 1) split_tc_kernel(const LaunchArgs a) {
  split_tc_body<C, PERSIST, FUSED>(a);
}

// The plain per-split kernel of a configuration with a pinned register budget
// (TcCfg MAXREG_ > 0).
template <class C>
__global__ void __launch_bounds__(C::THREADS) __maxnreg__(C::MAXREG) split_tc_kernel_pinned(const LaunchArgs a) {
  split_tc_body<C, false, false>(a);
}

// ================================================================ merge kernel

constexpr int kMergeWarps = 8;        // warps of a few-rows merge block
constexpr int kMergeFewSlots = 16;    // a row with at most this many partial slots: one warp
constexpr int kMergeBatchWide = 20;   // slots per warp per round trip when a row has 64 < S <= 160
constexpr int kMergeStagedRows = 64;  // rows (B * NH) from which the staged merge is used

// The merge for few rows (B * NH < kMergeStagedRows), where it is one short
// step in a chain of launches. One block per (32-dim slab, query head,
// sequence); lane = dim in the slab, warp w of W = partial slots w, w + W,
// ...; each warp issues the loads of kMergeBatch partials before using any and
// folds them into a running (max, sum, O); the W warp results are then
// combined the same way: M = max_s m_s, w_s = 2^(m_s - M),
// out = sum_s w_s O_s / sum_s w_s l_s. The first batch of loads goes out
// with the load of the row's length (every slot is in bounds); slots past
// the row's active splits are masked once the length has arrived.
template <int kMergeBatch, int kMergeWarps>  // partials whose loads one warp issues together; warps
__global__ void __launch_bounds__(kMergeWarps * 32) merge_kernel(const LaunchArgs a) {
  __shared__ float sacc[kMergeWarps][32];
  __shared__ float sl[kMergeWarps];
  __shared__ float sm[kMergeWarps];
  const int slab = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Dependents are released after the wait, not before: letting the next
  // split grid become resident while this layer's split grid still streams
  // cost the small-band ring 0.6 us per layer on GB300 (its early L2
  // requests compete with this layer's reads), more than it gained on MQA.
  grid_dependency_wait();
  grid_launch_dependents();
  const int len_b = a.lens[b];
  const int CS = a.cluster;
  const int nslots = a.num_splits / CS;  // one partial per block, or per cluster of blocks
  const size_t row = static_cast<size_t>(b) * a.NH + h;
  const float2* ml = reinterpret_cast<const float2*>(a.ws_ml + row * nslots * 2);
  const int d = slab * 32 + lane;
  const float* ob = a.ws_o + row * nslots * a.HS + d;
  float2 mlv[kMergeBatch];
  float ov[kMergeBatch];
#pragma unroll
  for (int u = 0; u < kMergeBatch; ++u) {
    const int s = warp + kMergeWarps * u;
    mlv[u] = s < nslots ? ml[s] : make_float2(kNegInf, 0.f);
    ov[u] = s < nslots ? ob[static_cast<size_t>(s) * a.HS] : 0.f;
  }
  int lo;
  const int band = band_of(len_b, a.capacity, a.window, false, &lo);
  const int chunk = chunk_of(band, a.num_splits, a.granule);
  const int act = a.tile_stride > 0 ? min(a.num_splits, (band + a.tile_stride - 1) / a.tile_stride)
                                    : active_splits(band, chunk);
  const int ns = (act + CS - 1) / CS;
  float mw = kNegInf, lw = 0.f, acc = 0.f;
  for (int s0 = warp; s0 < ns; s0 += kMergeWarps * kMergeBatch) {
    if (s0 != warp) {
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        const int s = s0 + kMergeWarps * u;
        mlv[u] = s < ns ? ml[s] : make_float2(kNegInf, 0.f);
        ov[u] = s < ns ? ob[static_cast<size_t>(s) * a.HS] : 0.f;
      }
    } else {
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        if (s0 + kMergeWarps * u >= ns) {
          mlv[u] = make_float2(kNegInf, 0.f);
          ov[u] = 0.f;
        }
      }
    }
    float bm = kNegInf;
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) bm = fmaxf(bm, mlv[u].x);
    const float mn = fmaxf(mw, bm);
    if (mn == kNegInf) continue;  // nothing but padding
    const float sc = exp2f(mw - mn);  // 0 while mw is still -inf
    lw *= sc;
    acc *= sc;
#pragma unroll
    for (int u = 0; u < kMergeBatch; ++u) {
      const float w = exp2f(mlv[u].x - mn);  // 0 for padding
      lw += w * mlv[u].y;
      acc += w * ov[u];
    }
    mw = mn;
  }
  sacc[warp][lane] = acc;
  if (lane == 0) {
    sl[warp] = lw;
    sm[warp] = mw;
  }
  __syncthreads();
  if (warp == 0) {
    float M = kNegInf;
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) M = fmaxf(M, sm[w]);
    float t = 0.f, L = 0.f;
    if (M != kNegInf) {
#pragma unroll
      for (int w = 0; w < kMergeWarps; ++w) {
        const float c = exp2f(sm[w] - M);
        t += c * sacc[w][lane];
        L += c * sl[w];
      }
    }
    const float val = ns > 0 ? t / L : 0.f;
    a.out[row * a.HS + d] = f32_to_bf16_bits(val);
    if (a.out_f32) a.out_f32[row * a.HS + d] = val;
  }
}

constexpr int kMergeDims = 64;        // head dims per merge block (one per thread, two threads per dim)
constexpr int kMergeThreads = 128;
constexpr int kMergeStageMax = 256;   // partial slots staged in shared memory at once

// Shared memory of a merge block: up to kMergeStageMax slots of 64 fp32 dims.
inline size_t merge_smem_bytes(int slots) {
  return static_cast<size_t>(std::min(slots, kMergeStageMax)) * kMergeDims * sizeof(float);
}

// Block-wide reductions of the merge block (every thread gets the result).
__device__ __forceinline__ float merge_block_max(float v, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < kMergeThreads / 32; ++w) r = fmaxf(r, red[w]);
  __syncthreads();
  return r;
}

__device__ __forceinline__ float merge_block_sum(float v, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = 0.f;
#pragma unroll
  for (int w = 0; w < kMergeThreads / 32; ++w) r += red[w];  // fixed order
  __syncthreads();
  return r;
}

// The merge for many rows (B * NH >= kMergeStagedRows).
// One block per (64-dim chunk, query head, sequence). Every one of the row's
// S / cluster slots holds a partial (a split with an empty slice writes
// O = 0, m = -inf, l = 0), so the merge needs no length. Per stage of up to
// kMergeStageMax slots, one bulk copy per slot brings the slot's 64 dims of
// O into shared memory while the threads load the slots' (m, l):
// M = max_s m_s, w_s = 2^(m_s - M), L = sum_s w_s l_s; then each thread sums
// w_s O_s over half of the slots for its dim, and out = sum / L. Stages
// combine online (rescaled by 2^(M_old - M_new)), so one memory round trip
// serves up to 256 partials. A row whose partials are all empty (len == 0)
// is 0; a NaN in any m or l makes the row NaN; a NaN in O reaches its dim.
__global__ void __launch_bounds__(kMergeThreads) merge_staged_kernel(const LaunchArgs a) {
  extern __shared__ __align__(128) float sO[];  // [stage][kMergeDims]
  __shared__ float sW[kMergeStageMax];
  __shared__ float sRed[kMergeThreads / 32];
  __shared__ float sHalf[kMergeDims];
  __shared__ __align__(8) uint64_t bar;
  const int tid = threadIdx.x;
  const int h = blockIdx.y, b = blockIdx.z, d0 = blockIdx.x * kMergeDims;
  const uint32_t bar_a = smem_u32(&bar);
  if (tid == 0) {
    mbar_init(bar_a, 1);
    fence_mbar_init();
  }
  __syncthreads();
  grid_dependency_wait();
  grid_launch_dependents();
  const int ns = a.num_splits / a.cluster;  // one partial per block, or per cluster of blocks
  const size_t row = static_cast<size_t>(b) * a.NH + h;
  const float* src = a.ws_o + row * ns * a.HS + d0;
  const float2* ml = reinterpret_cast<const float2*>(a.ws_ml) + row * ns;
  const int dim = tid % kMergeDims, half = tid / kMergeDims;

  float M = kNegInf, L = 0.f, acc = 0.f;
  bool nan_ml = false, failed = false;
  for (int base = 0, stage = 0; base < ns; base += kMergeStageMax, ++stage) {
    const int cnt = min(kMergeStageMax, ns - base);
    if (tid == 0) mbar_arrive_expect_tx(bar_a, static_cast<uint32_t>(cnt) * kMergeDims * 4);
    for (int s = tid; s < cnt; s += kMergeThreads)
      bulk_g2s(smem_u32(sO + s * kMergeDims), src + static_cast<size_t>(base + s) * a.HS, kMergeDims * 4, bar_a);
    // this stage's (m, l): two slots per thread
    float2 v[kMergeStageMax / kMergeThreads];
    float mx = kNegInf;
#pragma unroll
    for (int k = 0; k < kMergeStageMax / kMergeThreads; ++k) {
      const int s = tid + k * kMergeThreads;
      v[k] = s < cnt ? ml[base + s] : make_float2(kNegInf, 0.f);
      nan_ml |= isnan(v[k].x) || isnan(v[k].y);
      mx = fmaxf(mx, v[k].x);
    }
    const float Mn = fmaxf(M, merge_block_max(mx, sRed));
    float ls = 0.f;
#pragma unroll
    for (int k = 0; k < kMergeStageMax / kMergeThreads; ++k) {
      const int s = tid + k * kMergeThreads;
      const float w = Mn == kNegInf ? 0.f : exp2f(v[k].x - Mn);  // 0 for empty partials
      if (s < cnt) sW[s] = w;
      ls += w * v[k].y;
    }
    const float sc = M == kNegInf ? 0.f : exp2f(M - Mn);  // rescales the earlier stages
    L = L * sc + merge_block_sum(ls, sRed);               // (its barriers also publish sW)
    acc *= sc;
    M = Mn;
    mbar_wait(bar_a, stage & 1, failed);
    for (int s = half; s < cnt; s += 2) acc += sW[s] * sO[s * kMergeDims + dim];
    __syncthreads();  // the stage's buffers are free before the next copies
  }
  if (half == 1) sHalf[dim] = acc;
  const bool any_nan = __syncthreads_or(nan_ml) != 0;
  if (half == 0) {
    acc += sHalf[dim];
    const float val = any_nan ? __int_as_float(0x7fc00000) : (M == kNegInf ? 0.f : acc / L);
    a.out[row * a.HS + d0 + dim] = f32_to_bf16_bits(val);
    if (a.out_f32) a.out_f32[row * a.HS + d0 + dim] = val;
  }
}

// ================================================================ dispatch

// Launch with programmatic stream serialization allowed, so this kernel's
// blocks may be scheduled while the previous kernel on the stream drains; the
// kernels above wait (griddepcontrol.wait) before touching any input.
template <class... KArgs, class... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       int cluster, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The same with every block of the grid resident at once (a cooperative
// launch: the driver refuses a grid that cannot be), for kernels whose blocks
// wait on one another.
template <class... KArgs, class... Args>
cudaError_t launch_pdl_cooperative(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                   cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg{};
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
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Kernel attributes are set once per (kernel, device): the values never
// change, and the driver call would otherwise sit on every launch's host path.
template <auto Kernel>
cudaError_t smem_attr_once(int bytes) {
  static std::atomic<unsigned long long> done{0};  // bit d: set on device d
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

template <auto Kernel>
cudaError_t cluster_attr_once() {
  static std::atomic<unsigned long long> done{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

template <class C>
cudaError_t launch_tc(const LaunchArgs& a, cudaStream_t stream) {
  static_assert(C::SMEM <= 227 * 1024, "shared memory budget");
  cudaError_t e = smem_attr_once<split_tc_kernel<C>>(static_cast<int>(C::SMEM));
  if (e != cudaSuccess) return e;
  if (a.cluster > 8) {
    e = cluster_attr_once<split_tc_kernel<C>>();
    if (e != cudaSuccess) return e;
  }
  if (a.persistent > 0) {
    e = smem_attr_once<split_tc_kernel<C, true>>(static_cast<int>(C::SMEM));
    if (e != cudaSuccess) return e;
    return launch_pdl(split_tc_kernel<C, true>, dim3(a.persistent), dim3(C::THREADS), C::SMEM, stream, 1, a);
  }
  if (a.fused == kFusedGroup) {
    e = smem_attr_once<split_tc_kernel<C, false, kFusedGroup>>(static_cast<int>(C::SMEM));
    if (e != cudaSuccess) return e;
    return launch_pdl_cooperative(split_tc_kernel<C, false, kFusedGroup>, dim3(a.num_splits, a.NKV, a.B),
                                  dim3(C::THREADS), C::SMEM, stream, a);
  }
  if (a.fused) {
    e = smem_attr_once<split_tc_kernel<C, false, kFusedLast>>(static_cast<int>(C::SMEM));
    if (e != cudaSuccess) return e;
    return launch_pdl(split_tc_kernel<C, false, kFusedLast>, dim3(a.num_splits, a.NKV, a.B), dim3(C::THREADS),
                      C::SMEM, stream, 1, a);
  }
  dim3 grid(a.num_splits, a.NKV, a.B);
  if constexpr (C::MAXREG > 0) {
    if (a.cluster == 1) {
      e = smem_attr_once<split_tc_kernel_pinned<C>>(static_cast<int>(C::SMEM));
      if (e != cudaSuccess) return e;
      return launch_pdl(split_tc_kernel_pinned<C>, grid, dim3(C::THREADS), C::SMEM, stream, 1, a);
    }
  }
  return launch_pdl(split_tc_kernel<C>, grid, dim3(C::THREADS), C::SMEM, stream, a.cluster, a);
}

template <class C>
cudaError_t occupancy_tc(int* ctas) {
  if constexpr (C::MAXREG > 0) {
    cudaError_t e = smem_attr_once<split_tc_kernel_pinned<C>>(static_cast<int>(C::SMEM));
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, split_tc_kernel_pinned<C>, C::THREADS, C::SMEM);
  }
  cudaError_t e = smem_attr_once<split_tc_kernel<C>>(static_cast<int>(C::SMEM));
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, split_tc_kernel<C>, C::THREADS, C::SMEM);
}

// Tile configurations (measured on GB300, per head dim): 8 groups of 2 KB per
// tensor per stage (about 33 KB of K+V), three stages; G <= 8 or G <= 16
// query rows per group. The d128 and d256 tiles for G <= 8 and the d512 tiles
// fit two blocks per SM (100-111 KB each); the d64 tiles and the 16-row d128
// and d256 tiles (118-139 KB) fit one. Head dims 256 and 512 use eight
// consumer warps (shorter per-warp dependency chains; the one-block-per-SM
// MQA grids gained most). The head-dim-512, 16-row tile planned with one block
// per SM uses 4 KB groups: 66 KB stages, ~218 KB of shared memory.
using Tc64x1 = TcCfg<64, 1, 4, 3>;
using Tc64x2 = TcCfg<64, 2, 4, 3>;
using Tc128x1 = TcCfg<128, 1, 4, 3>;
using Tc128x2 = TcCfg<128, 2, 4, 3>;
// The head-dim-256 tile for up to 8 query rows (the sliding ring) copies 4 KB
// groups (64-position tiles) through two stages: the ring's band becomes 16
// one-tile splits per KV head instead of 32 of 32 positions (measured on
// GB300, us per layer: 6.14 with 2 KB groups in three stages, 6.04 with 4 KB
// groups in three, 5.99 in two). When the plan gives every split at most one
// tile, a one-stage instance serves it (half the shared memory, 5.84 against
// 6.04 on the same box); a split with more tiles would wait for each copy.
using Tc256x1 = TcCfg<256, 1, 8, 2, 4096>;
using Tc256x1s = TcCfg<256, 1, 8, 1, 4096>;
using Tc256x2 = TcCfg<256, 2, 8, 3>;
using Tc512x1 = TcCfg<512, 1, 4, 3>;  // a 16-position tile has 8 x 16 softmax slots
// The head-dim-512 bf16 tiles stream through two stages, not three (measured
// on GB300, us per layer: MQA 32k 19.25 -> 18.9, MQA 4k 8.83 -> 8.63 on the
// one-block-per-SM tile; MQA long 166.0 -> 163.8 on the two-blocks-per-SM
// tile): the copies of one stage cover a tile's math, and the smaller block
// leaves the SM more L1.
using Tc512x2 = TcCfg<512, 2, 8, 2, 2048, false, 96>;      // two blocks per SM (long MQA bands)
using Tc512x2w = TcCfg<512, 2, 8, 2, 4096, false, 96>;  // one block per SM, 4 KB copies
// E4M3 caches: a block's copy rate is set by the number of bulk copies it
// issues, so 2 KB E4M3 groups (the positions of a 4 KB bf16 group) in a
// two-stage ring, except head dim 256 (small sliding bands), where 1 KB groups
// in four stages keep a split near one tile. The head-dim-512, 16-row tile
// takes eight consumer warps when the grid is one block per SM and four
// otherwise (two blocks per SM share the issue slots).
using Tc64x1f = TcCfg<64, 1, 2, 2, 4096, true>;  // two consumer warps: 32 dims each
using Tc64x2f = TcCfg<64, 2, 2, 2, 4096, true>;
using Tc128x1f = TcCfg<128, 1, 4, 2, 4096, true>;
using Tc128x2f = TcCfg<128, 2, 4, 2, 4096, true>;
// The E4M3 ring tile: 2 KB E4M3 groups (64 positions) in two stages, like
// the bf16 one (measured on GB300, E4M3 ring 6.66 -> 6.35-6.39 us per layer
// against 1 KB groups in four stages).
using Tc256x1f = TcCfg<256, 1, 8, 2, 4096, true>;
using Tc256x2f = TcCfg<256, 2, 8, 4, 2048, true>;
using Tc512x1f = TcCfg<512, 1, 4, 2, 4096, true>;
using Tc512x2f = TcCfg<512, 2, 4, 2, 4096, true>;
using Tc512x2f8 = TcCfg<512, 2, 8, 2, 4096, true, 96>;  // one block per SM
// Head dims 64 and 128 with short bands (the plan's whole-tile splits): 1 KB
// E4M3 groups in four stages, half the default tile, so a short band spreads
// over twice as many blocks.
using Tc64x1fs = TcCfg<64, 1, 2, 4, 2048, true>;
using Tc64x2fs = TcCfg<64, 2, 2, 4, 2048, true>;
using Tc128x1fs = TcCfg<128, 1, 4, 4, 2048, true>;
using Tc128x2fs = TcCfg<128, 2, 4, 4, 2048, true>;

template <template <class> class Fn, class... Args>
cudaError_t with_tc_cfg(int HS, int G, int group_bytes, bool kv8, int warps, bool one_tile, Args&&... args) {
  const bool two = G > 8;
  if (kv8) {
    switch (HS) {
      case 64:
        if (group_bytes == 1024) return two ? Fn<Tc64x2fs>::run(args...) : Fn<Tc64x1fs>::run(args...);
        return two ? Fn<Tc64x2f>::run(args...) : Fn<Tc64x1f>::run(args...);
      case 128:
        if (group_bytes == 1024) return two ? Fn<Tc128x2fs>::run(args...) : Fn<Tc128x1fs>::run(args...);
        return two ? Fn<Tc128x2f>::run(args...) : Fn<Tc128x1f>::run(args...);
      case 256: return two ? Fn<Tc256x2f>::run(args...) : Fn<Tc256x1f>::run(args...);
      case 512:
        if (!two) return Fn<Tc512x1f>::run(args...);
        return warps == 8 ? Fn<Tc512x2f8>::run(args...) : Fn<Tc512x2f>::run(args...);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (HS) {
    case 64: return two ? Fn<Tc64x2>::run(args...) : Fn<Tc64x1>::run(args...);
    case 128: return two ? Fn<Tc128x2>::run(args...) : Fn<Tc128x1>::run(args...);
    case 256:
      if (two) return Fn<Tc256x2>::run(args...);
      return one_tile ? Fn<Tc256x1s>::run(args...) : Fn<Tc256x1>::run(args...);
    case 512:
      if (!two) return Fn<Tc512x1>::run(args...);
      return group_bytes >= 4096 ? Fn<Tc512x2w>::run(args...) : Fn<Tc512x2>::run(args...);
    default: return cudaErrorInvalidValue;
  }
}

template <class C>
cudaError_t max_cluster_tc(int* cluster) {
  cudaError_t e = cudaFuncSetAttribute(split_tc_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(C::SMEM));
  if (e != cudaSuccess) return e;
  const bool nonportable =
      cudaFuncSetAttribute(split_tc_kernel<C>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) == cudaSuccess;
  if (!nonportable) cudaGetLastError();
  for (int cs = nonportable ? 16 : 8; cs >= 2; cs /= 2) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(cs, 1, 1);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, split_tc_kernel<C>, &cfg) == cudaSuccess && n > 0) {
      *cluster = cs;
      return cudaSuccess;
    }
    cudaGetLastError();
  }
  *cluster = 1;
  return cudaSuccess;
}

template <class C>
struct MaxClusterFn {
  static cudaError_t run(int* cluster) { return max_cluster_tc<C>(cluster); }
};

template <class C>
struct LaunchFn {
  static cudaError_t run(const LaunchArgs& a, cudaStream_t s) { return launch_tc<C>(a, s); }
};
template <class C>
struct OccFn {
  static cudaError_t run(int* ctas) { return occupancy_tc<C>(ctas); }
};
template <class C>
struct TileFn {
  static cudaError_t run(int* t) {
    *t = C::T;
    return cudaSuccess;
  }
};

}  // namespace

int tc_short_tile_positions(int HS) {
  switch (HS) {
    case 64: return Tc64x1fs::T;
    case 128: return Tc128x1fs::T;
    default: return 0;
  }
}

int tc_tile_positions(int HS, bool kv8) {
  switch (HS) {
    case 64: return kv8 ? Tc64x1f::T : Tc64x1::T;
    case 128: return kv8 ? Tc128x1f::T : Tc128x1::T;
    case 256: return kv8 ? Tc256x1f::T : Tc256x1::T;
    case 512: return kv8 ? Tc512x1f::T : Tc512x1::T;
    default: return 16;
  }
}

// The whole-tile chunk granule of a kernel family: on the tensor-core path a
// block's time is its tiles' latency chain, so a split shorter than a tile
// costs as much as a full one while adding a partial to merge (measured on
// GB300: a 256-position band ran 23% faster as 4 one-tile splits than as 37
// splits of 7 positions). The SIMT kernel walks single positions.
int plan_granule(int path, int HS, bool kv8) { return path == FD_PATH_SIMT ? 1 : tc_tile_positions(HS, kv8); }

cudaError_t query_ctas_per_sm(int path, int HS, int G, bool kv8, int* ctas) {
  if (path == FD_PATH_SIMT) {
    const size_t sm = simt_smem_bytes(G, HS);
    cudaError_t e = cudaFuncSetAttribute(split_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(sm));
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, split_simt_kernel, kSimtThreads, sm);
  }
  return with_tc_cfg<OccFn>(HS, G, 2048, kv8, 0, false, ctas);
}

cudaError_t query_max_cluster(int HS, int G, bool kv8, int* cluster) {
  return with_tc_cfg<MaxClusterFn>(HS, G, 2048, kv8, 0, false, cluster);
}

cudaError_t launch_decode(const LaunchArgs& args, cudaStream_t stream) {
  const int G = args.NH / args.NKV;
  cudaError_t e;
  LaunchArgs a = args;
  a.tile_stride = 0;
  if (a.path == FD_PATH_TC && (a.window <= 0 || a.window >= a.capacity)) {
    e = with_tc_cfg<TileFn>(a.HS, G, a.group_bytes, a.kv8 != 0, a.consumer_warps, a.one_tile != 0, &a.tile_stride);
    if (e != cudaSuccess) return e;
  }
  if (a.path == FD_PATH_SIMT) {
    const size_t sm = simt_smem_bytes(G, a.HS);
    e = cudaFuncSetAttribute(split_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(sm));
    if (e != cudaSuccess) return e;
    dim3 grid(a.num_splits, a.NKV, a.B);
    e = launch_pdl(split_simt_kernel, grid, dim3(kSimtThreads), sm, stream, 1, a);
  } else if (a.path == FD_PATH_UMMA) {
    e = launch_umma(a, stream);
  } else {
    e = with_tc_cfg<LaunchFn>(a.HS, G, a.group_bytes, a.kv8 != 0, a.consumer_warps, a.one_tile != 0, a, stream);
  }
  // the split kernel wrote the output itself: one block / cluster per band, or
  // an in-launch merge (each group's last block, or the group step)
  if (e != cudaSuccess || a.num_splits == a.cluster || a.fused) return e;
  if (static_cast<long long>(a.B) * a.NH < kMergeStagedRows) {
    // one round trip of loads per warp: 8 slots each up to 64 partials per
    // row, 20 up to 160 behind a bf16 cache (measured on GB300, us per layer:
    // MQA 32k with 152 partials per row 19.7 -> 19.3; behind the E4M3 split
    // kernel the wide merge lost, 22.5 -> 27.4, so E4M3 keeps rounds of 8)
    dim3 mgrid(a.HS / 32, a.NH, a.B);
    const int ns = a.num_splits / a.cluster;
    if (!a.kv8 && ns > kMergeWarps * 8 && ns <= kMergeWarps * kMergeBatchWide)
      return launch_pdl(merge_kernel<kMergeBatchWide, kMergeWarps>, mgrid, dim3(kMergeWarps * 32), 0, stream, 1, a);
    // up to 16 slots: one warp, every slot's loads in one round trip
    // (measured in same-box A/Bs, us per layer: eight warps -> two, ring with
    // 16 partials 5.79 -> 5.73, Llama tiny 4.78 -> 4.67; two -> one, ring
    // 5.68 -> 5.58, tiny 4.70 -> 4.62; four warps were slower on the ring,
    // 5.99, and few warps lose where rows have many slots, MQA 32k 19.25 ->
    // 23.8 at two)
    if (ns <= kMergeFewSlots)
      return launch_pdl(merge_kernel<kMergeFewSlots, 1>, mgrid, dim3(32), 0, stream, 1, a);
    return launch_pdl(merge_kernel<8, kMergeWarps>, mgrid, dim3(kMergeWarps * 32), 0, stream, 1, a);
  }
  const size_t msmem = merge_smem_bytes(a.num_splits / a.cluster);
  e = smem_attr_once<merge_staged_kernel>(static_cast<int>(merge_smem_bytes(kMergeStageMax)));
  if (e != cudaSuccess) return e;
  dim3 mgrid(a.HS / kMergeDims, a.NH, a.B);
  return launch_pdl(merge_staged_kernel, mgrid, dim3(kMergeThreads), msmem, stream, 1, a);
}

cudaError_t set_wait_limit(unsigned long long ns) {
  const unsigned long long v = ns ? ns : 1000000000ull;
  return cudaMemcpyToSymbol(g_wait_limit_ns, &v, sizeof v);
}

cudaError_t read_and_clear_device_error(cudaStream_t stream, unsigned int* err) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  unsigned int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof v);
  if (e != cudaSuccess) return e;
  const unsigned int zero = 0;
  e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof zero);
  if (e != cudaSuccess) return e;
  *err = v;
  return read_and_clear_device_error_umma(err);
}

}  // namespace fd
