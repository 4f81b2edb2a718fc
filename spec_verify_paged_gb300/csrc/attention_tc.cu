// attention_tc.cu -- paged decode / speculative-verify attention on the
// fifth-generation tensor cores of sm_103a (tcgen05.mma, accumulators in
// tensor memory).
//
// What it computes is what attention.cu computes (pages: "KV cache & Flash
// Attention", sections "FlashAttention -- the tiling trick" and
// "PagedAttention"; "How speculative decoding doubles LLM speed", step 2;
// "How StreamingLLM stabilizes million-token streams via attention sinks",
// section "The StreamingLLM solution"): for every query row (b, i, h) the
// softmax of the scaled scores over its visible keys, times V, and the
// log-sum-exp.  This kernel serves bf16 caches with head_dim 128 when a kv
// head has several query rows (GQA group x q_len).
//
// Orientation.  Keys are the M = 128 dimension of the MMA (one tile = 8
// pages), the N <= 32 query rows of a group are the N dimension:
//   S^T [128 keys x N]  = K_tile [128 x 128 d] . Q^T         A = K, K-major
//   O_t^T [128 d x N]   = V_tile^T [128 d x 128 keys] . P^T  A = V, MN-major
// so a 20-row verify group costs a 32-column MMA instead of a 128-row one,
// and both K and V feed the tensor core straight from the TMA-written
// 128-byte-swizzled tiles.  Accumulators live in tensor memory (TMEM):
// two S buffers and two O buffers of N columns, double-buffered by tile.
//
// Warp roles (192 threads, one CTA per SM):
//   warps 0-3  softmax and epilogue.  Thread k reads TMEM lane k: key k of
//              the tile for S, head dim k for O.  Column statistics (row
//              max and sum over the tile's keys) use a transposing warp
//              butterfly and four-warp exchange in shared memory; P goes
//              back to shared memory as bf16 in the MMA's swizzled layout.
//              Each tile's O_t is folded into registers (o = o * alpha +
//              O_t) while the tensor core works on the next tile.
//   warp 4     producer: block table, 2-D TMA copies of 8 pages' K and V
//              into a 3-stage ring.
//   warp 5     one thread issues tcgen05.mma / tcgen05.commit.
// Scheduling, split tickets and the merge are shared with attention.cu
// (attn_common.cuh).  Every wait is bounded; a timeout raises
// SVP_DEV_TIMEOUT and every role drains what it started before the CTA
// frees its tensor memory.
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "attn_common.cuh"

namespace svp {

static __device__ unsigned int g_status_attn_tc;

namespace {

constexpr int kD = 128;
constexpr int kTilePages = 8;
constexpr int kTileKeys = kTilePages * kBlockSize;  // the MMA's M
constexpr int kHalfBytes = kTileKeys * 128;  // 64 columns x 128 keys, bf16
constexpr int kTileBytes = 2 * kHalfBytes;   // one K (or V) tile: 32 KB
constexpr int kStages = 3;
constexpr int kSoftWarps = 4;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kTcThreads = 32 * 6;
constexpr int kPageTxBytes = 2 * 2 * kBoxBytes;  // K and V, two boxes each
constexpr int kTcBatchCap = 1024;  // sequences per launch (prefix in smem)

template <int N>
struct TcSmem {
  alignas(1024) unsigned char k[kStages][kTileBytes];
  alignas(1024) unsigned char v[kStages][kTileBytes];
  alignas(1024) unsigned char q[N * kD * 2];
  alignas(1024) unsigned char pb[2][N * kTileKeys * 2];
  alignas(16) float red_m[kSoftWarps][N];
  alignas(16) float red_l[2][kSoftWarps][N];
  alignas(16) float mu[N];        // the max each tile's p was taken against
  alignas(16) float alpha[2][N];  // rescale of the running state by a tile
  float row_inv[N];
  float row_m[N], row_w[N];
  UnitInfo unit[kUnitRing];
  int stage_mask[kStages];  // bit k: page k of the tile was copied
  uint64_t full[kStages], empty[kStages];
  uint64_t s_full[2], p_full[2], o_full[2], o_free[2];
  uint64_t q_full;
  uint64_t ufull[kUnitRing], uempty[kUnitRing];
  uint64_t epi;
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag, is_last, total_pages, n_ctas;
  int prefix[1];  // [batch + 1], dynamic
};

template <int N>
constexpr size_t tc_smem_bytes(int batch) {
  return sizeof(TcSmem<N>) + sizeof(int) * (size_t)batch + 1024;
}
static_assert(tc_smem_bytes<32>(kTcBatchCap + 1) <= 227 * 1024,
              "shared memory of a 32-row CTA");
static_assert(tc_smem_bytes<16>(kTcBatchCap + 1) <= 227 * 1024,
              "shared memory of a 16-row CTA");

__device__ __forceinline__ void raise_tc(unsigned f) {
  atomicOr(&g_status_attn_tc, f);
}

// ---- tcgen05 wrappers ----

// Shared-memory matrix descriptor, 128-byte swizzle: start address, leading
// and stride byte offsets (16-byte units), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr, uint32_t lbo,
                                               uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) |
         ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) |
         (2ull << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulate, bf16 A and B,
// A / B major-ness (0 = K-major, 1 = MN-major), N >> 3, M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n, int a_mn,
                                                  int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) |
         ((uint32_t)b_mn << 16) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a, uint64_t b,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives on `bar` once every tcgen05.mma this thread issued has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 "
      "[%0];" ::"r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// N consecutive 32-bit columns of this thread's TMEM lane.
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t addr, float (&v)[N]);

template <>
__device__ __forceinline__ void tmem_ld<16>(uint32_t addr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,"
      "%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
        "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]),
        "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(addr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

template <>
__device__ __forceinline__ void tmem_ld<32>(uint32_t addr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,"
      "%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,"
      "%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
        "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]),
        "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
        "=r"(r[30]), "=r"(r[31])
      : "r"(addr));
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Column reduction over the 32 keys (lanes) of a warp: each lane holds N
// columns; a transposing butterfly halves the columns each step, so lane l
// ends with column col_of(l) of the warp's max (or sum) after N-1 shuffles.
template <int N>
__device__ __forceinline__ int col_of(int lane) {
  return N == 32 ? lane : lane >> 1;
}

template <int N, bool MAX>
__device__ __forceinline__ float col_reduce(const float (&x)[N], int lane) {
  static_assert(N == 16 || N == 32, "16 or 32 columns");
  float v[N];
#pragma unroll
  for (int i = 0; i < N; ++i) v[i] = x[i];
#pragma unroll
  for (int h = N / 2, off = 16; h >= 1; h >>= 1, off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < h; ++i) {
      const float send = upper ? v[i] : v[i + h];
      const float keep = upper ? v[i + h] : v[i];
      const float got = __shfl_xor_sync(kFull, send, off);
      v[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  if (N == 16) {  // lanes l and l ^ 1 hold halves of the same column
    const float got = __shfl_xor_sync(kFull, v[0], 1);
    v[0] = MAX ? fmaxf(v[0], got) : v[0] + got;
  }
  return v[0];
}

// Byte offset of element (row n, column k) of an [N rows x 128 columns]
// bf16 operand in the K-major 128-byte-swizzled layout: two 64-column
// halves, each [N][128 B], 16-byte chunks XOR-ed with the row mod 8.
template <int N>
__device__ __forceinline__ uint32_t kmajor_off(int n, int k) {
  return (uint32_t)((k >> 6) * (N * 128) + n * 128 +
                    ((((k & 63) >> 3) ^ (n & 7)) << 4) + (k & 7) * 2);
}

}  // namespace

// --------------------------------------------------------------------------
// the kernel
// --------------------------------------------------------------------------
template <int N>
__global__ void __launch_bounds__(kTcThreads, 1)
    paged_attention_tc_kernel(const AttnParams p,
                              const __grid_constant__ TensorMaps tm) {
  extern __shared__ unsigned char smem_raw[];
  TcSmem<N> &sm = *reinterpret_cast<TcSmem<N> *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr uint32_t kTmemCols = 4 * N;  // S[2], O[2]
  constexpr uint32_t kIdescS = idesc_bf16(kTileKeys, N, 0, 0);
  constexpr uint32_t kIdescO = idesc_bf16(kD, N, 1, 0);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int groups_per_seq = p.num_kv_heads * p.n_rg;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int b2 = 0; b2 < 2; ++b2) {
      mbar_init(&sm.s_full[b2], 1);
      mbar_init(&sm.p_full[b2], kSoftWarps);
      mbar_init(&sm.o_full[b2], 1);
      mbar_init(&sm.o_free[b2], kSoftWarps);
    }
    mbar_init(&sm.q_full, kSoftWarps);
    for (int u = 0; u < kUnitRing; ++u) {
      mbar_init(&sm.ufull[u], 1);
      mbar_init(&sm.uempty[u], 2);  // softmax warps and the MMA thread
    }
    mbar_init(&sm.epi, kSoftWarps);
    mbar_init(&sm.drain, 1);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    asm volatile(
        "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
            smem_u32(&sm.tmem_base)),
        "r"(kTmemCols)
        : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::
                     : "memory");
  }
  if (warp == 0) {
    const int run = build_prefix(p, sm.prefix, groups_per_seq, lane,
                                 &g_status_attn_tc);
    if (lane == 0) {
      sm.total_pages = run;
      sm.n_ctas = working_ctas(run, p.min_pages);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const int total_pages = sm.total_pages;
  const int n_ctas = sm.n_ctas;
  const int range_begin = slice_begin(blockIdx.x, total_pages, n_ctas);
  const int range_end = blockIdx.x < n_ctas
                            ? slice_begin(blockIdx.x + 1, total_pages, n_ctas)
                            : total_pages;

  if (warp == kProducerWarp) {
    // ======================= producer warp =======================
    int c = 0;   // tiles issued so far
    int us = 0;  // segments published so far
    bool ok = true;
    int pos = range_begin;
    while (true) {
      const int slot = us % kUnitRing;
      if (lane == 0)
        ok = mbar_wait(&sm.uempty[slot], ((us / kUnitRing) & 1) ^ 1);
      ok = __shfl_sync(kFull, ok, 0) && !sm.abort_flag;
      if (!ok) break;
      if (pos >= range_end) {
        if (lane == 0) {
          sm.unit[slot].valid = 0;
          mbar_arrive(&sm.ufull[slot]);
        }
        break;
      }
      const UnitInfo seg =
          decode_segment(p, sm.prefix, groups_per_seq, pos, range_begin,
                         range_end, total_pages, n_ctas);
      if (lane == 0) {
        sm.unit[slot] = seg;
        mbar_arrive(&sm.ufull[slot]);
      }
      const int n_pages = seg.n_pages;
      for (int k0 = 0; k0 < n_pages && ok; k0 += kTableChunk) {
        // block-table entries of the next 128 pages, one coalesced load each
        int phys[kTableChunk / 32];
#pragma unroll
        for (int k4 = 0; k4 < kTableChunk / 32; ++k4) {
          const int k = k0 + k4 * 32 + lane;
          phys[k4] = -1;
          if (k < n_pages)
            phys[k4] = __ldg(p.block_table + (size_t)seg.b * p.max_blocks +
                             logical_block(seg, seg.page0 + k));
        }
        const int kend = min(k0 + kTableChunk, n_pages);
        for (int t0 = k0; t0 < kend; t0 += kTilePages) {
          // tiles start at multiples of 8 pages of the segment; lane kk < 8
          // copies page t0 + kk, whose entry sits in lane (t0-k0)%32 + kk
          const int npg = min(kTilePages, n_pages - t0);
          const int k4 = (t0 - k0) >> 5;
          const int src = k4 == 0 ? phys[0] : k4 == 1 ? phys[1]
                        : k4 == 2 ? phys[2] : phys[3];
          const int ph = __shfl_sync(kFull, src, ((t0 - k0) & 31) + (lane & 7));
          const bool mine = lane < npg;
          const bool good = mine && ph >= 0 && ph < p.num_blocks;
          if (mine && !good) raise_tc(SVP_DEV_BAD_BLOCK_ID);
          const unsigned mask = __ballot_sync(kFull, good) & 0xffu;
          const int s = c % kStages;
          if (lane == 0) {
            if (!mbar_wait(&sm.empty[s], ((c / kStages) & 1) ^ 1)) {
              ok = false;
            } else {
              sm.stage_mask[s] = (int)mask;
              if (mask)
                mbar_arrive_expect_tx(&sm.full[s], __popc(mask) * kPageTxBytes);
              else
                mbar_arrive(&sm.full[s]);
            }
          }
          ok = __shfl_sync(kFull, ok, 0);  // also orders the copies after it
          if (!ok) break;
          if (good) {
            const int y = (ph * p.num_kv_heads + seg.g) * kBlockSize;
#pragma unroll
            for (int bx = 0; bx < 2; ++bx) {
              tma_load_2d(sm.k[s] + bx * kHalfBytes + lane * kBoxBytes, &tm.k,
                          bx * kBoxElems, y, &sm.full[s]);
              tma_load_2d(sm.v[s] + bx * kHalfBytes + lane * kBoxBytes, &tm.v,
                          bx * kBoxElems, y, &sm.full[s]);
            }
          }
          ++c;
        }
      }
      if (!ok) break;
      pos += n_pages;
      ++us;
    }
    if (!ok && lane == 0) {
      // give up: flag it, then wait (bounded) for copies still in flight
      raise_tc(SVP_DEV_TIMEOUT);
      sm.abort_flag = 1;
      for (int k = max(0, c - kStages); k < c; ++k)
        (void)mbar_wait(&sm.full[k % kStages], (k / kStages) & 1);
    }
  } else if (warp == kMmaWarp) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      bool ok = true;
      int c = 0, us = 0;
      int pend = -1, pend_npg = 0;  // the tile whose P V is not issued yet
      // O_t^T = V^T P^T over the tile's npg pages (16 keys per k-step)
      auto issue_pv = [&](int t, int npg) -> bool {
        const int b2 = t & 1;
        if (!mbar_wait(&sm.p_full[b2], (t >> 1) & 1)) return false;
        if (t >= 2 && !mbar_wait(&sm.o_free[b2], ((t - 2) >> 1) & 1))
          return false;
        tc_fence_after();
        const int s = t % kStages;
        const uint32_t va = smem_u32(sm.v[s]), pa = smem_u32(sm.pb[b2]);
        for (int ks = 0; ks < npg; ++ks) {
          // V as MN-major A: 64-dim halves kHalfBytes apart (leading byte
          // offset), 8-key groups 1024 B apart (stride byte offset)
          const uint64_t a = sw128_desc(va + ks * 2048, kHalfBytes, 1024);
          const uint64_t b =
              sw128_desc(pa + (ks >> 2) * (N * 128) + (ks & 3) * 32, 16, 1024);
          tc_mma(tmem + 2 * N + b2 * N, a, b, kIdescO, ks > 0 ? 1u : 0u);
        }
        tc_commit(&sm.empty[s]);
        tc_commit(&sm.o_full[b2]);
        return true;
      };
      while (ok) {
        const int slot = us % kUnitRing;
        if (!mbar_wait(&sm.ufull[slot], (us / kUnitRing) & 1)) {
          ok = false;
          break;
        }
        const UnitInfo ui = sm.unit[slot];
        mbar_arrive(&sm.uempty[slot]);
        if (!ui.valid || sm.abort_flag) break;
        const int tiles = (ui.n_pages + kTilePages - 1) / kTilePages;
        for (int tau = 0; tau < tiles; ++tau, ++c) {
          const int s = c % kStages, b2 = c & 1;
          if (!mbar_wait(&sm.full[s], (c / kStages) & 1)) { ok = false; break; }
          if (tau == 0) {
            // finish the previous segment before waiting for this one's Q
            if (pend >= 0 && !issue_pv(pend, pend_npg)) { ok = false; break; }
            pend = -1;
            if (!mbar_wait(&sm.q_full, us & 1)) { ok = false; break; }
          }
          tc_fence_after();
          // S^T = K Q^T: 8 k-steps of 16 head dims (32 B inside a 128-B row)
          const uint32_t ka = smem_u32(sm.k[s]), qa = smem_u32(sm.q);
#pragma unroll
          for (int ks = 0; ks < kD / 16; ++ks) {
            const uint64_t a =
                sw128_desc(ka + (ks >> 2) * kHalfBytes + (ks & 3) * 32, 16, 1024);
            const uint64_t b =
                sw128_desc(qa + (ks >> 2) * (N * 128) + (ks & 3) * 32, 16, 1024);
            tc_mma(tmem + b2 * N, a, b, kIdescS, ks > 0 ? 1u : 0u);
          }
          tc_commit(&sm.s_full[b2]);
          if (pend >= 0 && !issue_pv(pend, pend_npg)) { ok = false; break; }
          pend = c;
          pend_npg = min(kTilePages, ui.n_pages - tau * kTilePages);
        }
        ++us;
      }
      if (ok && pend >= 0) ok = issue_pv(pend, pend_npg);
      if (!ok) {
        raise_tc(SVP_DEV_TIMEOUT);
        sm.abort_flag = 1;
      }
      // every MMA issued has completed before tensor memory is freed
      tc_commit(&sm.drain);
      (void)mbar_wait(&sm.drain, 0);
    }
    __syncwarp();
  } else {
    // ======================= softmax warps =======================
    const int ctid = tid;  // key of the tile (S), head dim (O)
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    uint32_t epi_phase = 0;
    int c = 0, us = 0;
    bool aborted = false;
    // O of tile t: wait, read, release the buffer, fold into o
    auto fold_o = [&](int t, float (&o)[N]) -> bool {
      const int b2 = t & 1;
      const bool got = mbar_wait(&sm.o_full[b2], (t >> 1) & 1);
      if (!__all_sync(kFull, got)) return false;
      tc_fence_after();
      float ov[N];
      tmem_ld<N>(tmem + lane_base + 2 * N + b2 * N, ov);
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.o_free[b2]);
      const float4 *al = reinterpret_cast<const float4 *>(sm.alpha[b2]);
#pragma unroll
      for (int n4 = 0; n4 < N / 4; ++n4) {
        const float4 a = al[n4];
        o[4 * n4 + 0] = fmaf(o[4 * n4 + 0], a.x, ov[4 * n4 + 0]);
        o[4 * n4 + 1] = fmaf(o[4 * n4 + 1], a.y, ov[4 * n4 + 1]);
        o[4 * n4 + 2] = fmaf(o[4 * n4 + 2], a.z, ov[4 * n4 + 2]);
        o[4 * n4 + 3] = fmaf(o[4 * n4 + 3], a.w, ov[4 * n4 + 3]);
      }
      return true;
    };
    while (true) {
      const int slot = us % kUnitRing;
      const bool got =
          __all_sync(kFull, mbar_wait(&sm.ufull[slot], (us / kUnitRing) & 1));
      if (!got) { aborted = true; break; }
      const UnitInfo ui = sm.unit[slot];
      if (!ui.valid || sm.abort_flag) break;
      const int b = ui.b, g = ui.g, rg = ui.rg, L = ui.seq_len;
      const int t0 = L - p.q_len;
      const int vrows = min(N, p.rows - rg * N);

      // ---- Q of the group -> shared memory (rows past vrows are zero) ----
      for (int idx = ctid; idx < N * 16; idx += kSoftWarps * 32) {
        const int n = idx >> 4, ch = idx & 15;
        uint4 val = make_uint4(0u, 0u, 0u, 0u);
        if (n < vrows) {
          const int gr = rg * N + n;
          const int i = gr / p.group, h = g * p.group + gr % p.group;
          val = __ldg(reinterpret_cast<const uint4 *>(
                          static_cast<const uint16_t *>(p.q) +
                          (((size_t)b * p.q_len + i) * p.num_q_heads + h) * kD) +
                      ch);
        }
        *reinterpret_cast<uint4 *>(sm.q + kmajor_off<N>(n, ch * 8)) = val;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sm.q_full);

      float o[N];
#pragma unroll
      for (int n = 0; n < N; ++n) o[n] = 0.f;
      // running column statistics, kept by thread n < N for row n
      float m_run = -INFINITY, l_run = 0.f, alpha_prev = 1.f;
      const int tiles = (ui.n_pages + kTilePages - 1) / kTilePages;
      // first global row of this group: visibility bounds are row indices
      const int row0 = rg * N;
      for (int tau = 0; tau < tiles; ++tau, ++c) {
        const int s = c % kStages, b2 = c & 1;
        bool ok = mbar_wait(&sm.s_full[b2], (c >> 1) & 1);
        ok = ok && mbar_wait(&sm.full[s], (c / kStages) & 1);
        if (!__all_sync(kFull, ok)) { aborted = true; break; }
        tc_fence_after();
        float sv[N];
        tmem_ld<N>(tmem + lane_base + b2 * N, sv);
        tc_wait_ld();

        // ---- this thread's key ----
        const int kslot = ctid >> 4, r = ctid & 15;
        const int npg = min(kTilePages, ui.n_pages - tau * kTilePages);
        const bool loaded = ((sm.stage_mask[s] >> kslot) & 1) != 0;
        const int j =
            logical_block(ui, ui.page0 + tau * kTilePages + kslot) * kBlockSize + r;
        // visible to some row of the call: holds real data
        const bool in_union = loaded && j < L &&
                              (p.window == 0 || j < p.n_sink || j > t0 - p.window);
        if (kslot < npg && !in_union) {
          // p = 0 here, but 0 * NaN left in unused cache rows is still NaN
#pragma unroll
          for (int bx = 0; bx < 2; ++bx)
#pragma unroll
            for (int ch = 0; ch < 8; ++ch)
              *reinterpret_cast<uint4 *>(sm.v[s] + bx * kHalfBytes + ctid * 128 +
                                         ch * 16) = make_uint4(0u, 0u, 0u, 0u);
        }
        // rows n (of this group) that see key j: n in [nlo, nhi).  Row n is
        // query position i = (row0 + n) / group, at t0 + i.
        int nlo = 0, nhi = N;
        if (!in_union) {
          nlo = N;
        } else {
          if (j > t0) nlo = min(N, (j - t0) * p.group - row0);
          if (p.window != 0 && j >= p.n_sink) {
            const long long lim = (long long)(j + p.window - t0) * p.group - row0;
            nhi = lim < N ? (int)lim : N;
          }
        }
        const bool all_vis = __all_sync(kFull, nlo <= 0 && nhi >= N);
#pragma unroll
        for (int n = 0; n < N; ++n) {
          const float x = sv[n] * p.qscale;
          sv[n] = (all_vis || (n >= nlo && n < nhi)) ? x : -INFINITY;
        }

        // ---- column max over the tile's 128 keys ----
        const float cm = col_reduce<N, true>(sv, lane);
        if (N == 32 || (lane & 1) == 0) sm.red_m[warp][col_of<N>(lane)] = cm;
        if (!consumer_sync(&sm.epi, epi_phase, lane)) { aborted = true; break; }
        if (ctid < N) {
          const float mt = fmaxf(fmaxf(sm.red_m[0][ctid], sm.red_m[1][ctid]),
                                 fmaxf(sm.red_m[2][ctid], sm.red_m[3][ctid]));
          if (tau > 0) {
            const int pb2 = b2 ^ 1;
            l_run = fmaf(l_run, alpha_prev,
                         (sm.red_l[pb2][0][ctid] + sm.red_l[pb2][1][ctid]) +
                             (sm.red_l[pb2][2][ctid] + sm.red_l[pb2][3][ctid]));
          }
          const float m_new = fmaxf(m_run, mt);
          const float mu = m_new == -INFINITY ? 0.f : m_new;
          alpha_prev = ex2(m_run - mu);  // 0 while nothing was visible
          m_run = m_new;
          sm.mu[ctid] = mu;
          sm.alpha[b2][ctid] = alpha_prev;
        }
        if (!consumer_sync(&sm.epi, epi_phase, lane)) { aborted = true; break; }

        // ---- p = exp2(s - mu), column sums, P -> shared memory (bf16) ----
        {
          const float4 *mu4 = reinterpret_cast<const float4 *>(sm.mu);
#pragma unroll
          for (int n4 = 0; n4 < N / 4; ++n4) {
            const float4 m4 = mu4[n4];
            sv[4 * n4 + 0] = ex2(sv[4 * n4 + 0] - m4.x);
            sv[4 * n4 + 1] = ex2(sv[4 * n4 + 1] - m4.y);
            sv[4 * n4 + 2] = ex2(sv[4 * n4 + 2] - m4.z);
            sv[4 * n4 + 3] = ex2(sv[4 * n4 + 3] - m4.w);
          }
        }
        const float cs = col_reduce<N, false>(sv, lane);
        if (N == 32 || (lane & 1) == 0) sm.red_l[b2][warp][col_of<N>(lane)] = cs;
        unsigned char *pbuf = sm.pb[b2];
#pragma unroll
        for (int n = 0; n < N; ++n) {
          const __nv_bfloat16 h = __float2bfloat16_rn(sv[n]);
          *reinterpret_cast<__nv_bfloat16 *>(pbuf + kmajor_off<N>(n, ctid)) = h;
        }
        fence_proxy_async_smem();  // P and zeroed V rows -> tensor core
        tc_fence_before();         // S reads done before S is rewritten
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_full[b2]);

        // ---- fold the previous tile's O while this tile's P V runs ----
        if (tau > 0 && !fold_o(c - 1, o)) { aborted = true; break; }
      }
      if (aborted) break;
      if (!fold_o(c - 1, o)) { aborted = true; break; }
      // last tile's sums: every warp wrote them before its p_full arrival;
      // a barrier makes them visible to the row threads
      if (!consumer_sync(&sm.epi, epi_phase, lane)) { aborted = true; break; }

      // ---- epilogue ----
      const bool single = ui.f == ui.l;
      const size_t pslot = (size_t)(2 * blockIdx.x + ui.slot);
      if (ctid < N) {
        const int lb2 = (c - 1) & 1;
        l_run = fmaf(l_run, alpha_prev,
                     (sm.red_l[lb2][0][ctid] + sm.red_l[lb2][1][ctid]) +
                         (sm.red_l[lb2][2][ctid] + sm.red_l[lb2][3][ctid]));
        const float mu = m_run == -INFINITY ? 0.f : m_run;
        sm.row_inv[ctid] = l_run > 0.f ? 1.f / l_run : 0.f;
        const float lse2 = l_run > 0.f ? mu + log2f(l_run) : -INFINITY;
        if (ctid < vrows) {
          const int gr = row0 + ctid;
          if (single) {
            const int i = gr / p.group, h = g * p.group + gr % p.group;
            p.lse[((size_t)b * p.q_len + i) * p.num_q_heads + h] = lse2 * kLn2;
          } else {
            p.part_lse[pslot * N + ctid] = lse2;
          }
        }
      }
      if (!consumer_sync(&sm.epi, epi_phase, lane)) { aborted = true; break; }
#pragma unroll
      for (int n = 0; n < N; ++n) {
        if (n < vrows) {
          const float val = o[n] * sm.row_inv[n];
          if (single) {
            const int gr = row0 + n;
            const int i = gr / p.group, h = g * p.group + gr % p.group;
            store_out(static_cast<uint16_t *>(p.out) +
                          (((size_t)b * p.q_len + i) * p.num_q_heads + h) * kD +
                          ctid,
                      val);
          } else {
            p.part_o[(pslot * N + n) * kD + ctid] = val;
          }
        }
      }
      if (!single) {
        __threadfence();
        if (!consumer_sync(&sm.epi, epi_phase, lane)) { aborted = true; break; }
        if (ctid == 0)
          sm.is_last = take_ticket(p, (b * p.num_kv_heads + g) * p.n_rg + rg,
                                   ui.l - ui.f + 1);
        if (!consumer_sync(&sm.epi, epi_phase, lane)) { aborted = true; break; }
        if (sm.is_last) {
          __threadfence();
          // the P buffers are idle between segments: merge scratch
          if (!merge_partials<uint16_t, kD, N, kSoftWarps * 32>(
                  p, ui, total_pages, n_ctas,
                  reinterpret_cast<float *>(&sm.pb[0][0]),
                  (int)(sizeof(sm.pb) / sizeof(float)), sm.row_m, sm.row_w,
                  &sm.epi, epi_phase, ctid)) {
            aborted = true;
            break;
          }
        }
      }
      if (!consumer_sync(&sm.epi, epi_phase, lane)) { aborted = true; break; }
      if (ctid == 0) mbar_arrive(&sm.uempty[slot]);
      ++us;
    }
    if (aborted && lane == 0) {
      raise_tc(SVP_DEV_TIMEOUT);
      sm.abort_flag = 1;
    }
  }

  // no warp leaves while others may use the barriers; tensor memory is
  // freed once the MMA thread has seen its last MMA complete
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(
                     tmem),
                 "r"(kTmemCols)
                 : "memory");
}

// --------------------------------------------------------------------------
// host side
// --------------------------------------------------------------------------
static std::mutex g_tc_mu;
static std::map<std::tuple<int, const void *, size_t>, int> g_tc_occ;

static size_t tc_batch_bucket(int batch) {
  return (size_t)(batch + 255) / 256 * 256;
}

template <int N>
static int prepare_tc(int batch) {
  const size_t smem = tc_smem_bytes<N>((int)tc_batch_bucket(batch));
  auto kern = paged_attention_tc_kernel<N>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  const auto key = std::make_tuple(dev, (const void *)kern, smem);
  {
    std::lock_guard<std::mutex> lk(g_tc_mu);
    auto it = g_tc_occ.find(key);
    if (it != g_tc_occ.end()) return it->second;
  }
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return -1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kTcThreads,
                                                    smem) != cudaSuccess)
    return -1;
  if (n < 1) return -1;
  std::lock_guard<std::mutex> lk(g_tc_mu);
  g_tc_occ[key] = n;
  return n;
}

template <int N>
static cudaError_t launch_tc(const AttnParams &p, int grid, cudaStream_t st) {
  if (prepare_tc<N>(p.batch) < 0) return cudaErrorInvalidValue;
  const size_t smem = tc_smem_bytes<N>((int)tc_batch_bucket(p.batch));
  TensorMaps tm;
  memset(&tm, 0, sizeof tm);
  if (!make_kv_map(&tm.k, p.k_cache, p.num_blocks, p.num_kv_heads, kD) ||
      !make_kv_map(&tm.v, p.v_cache, p.num_blocks, p.num_kv_heads, kD))
    return cudaErrorInvalidValue;
  paged_attention_tc_kernel<N><<<grid, kTcThreads, smem, st>>>(p, tm);
  return cudaGetLastError();
}

int tc_batch_cap() { return kTcBatchCap; }

int attention_tc_ctas_per_sm(int rb, int batch) {
  const int n = rb == 16 ? prepare_tc<16>(batch) : prepare_tc<32>(batch);
  return n > 0 ? n : 1;
}

cudaError_t launch_attention_tc(const AttnParams &p, int grid,
                                cudaStream_t stream) {
  if (p.head_dim != kD || (p.rb != 16 && p.rb != 32) ||
      p.batch > kTcBatchCap)
    return cudaErrorInvalidValue;
  return p.rb == 16 ? launch_tc<16>(p, grid, stream)
                    : launch_tc<32>(p, grid, stream);
}

cudaError_t read_status_attention_tc(cudaStream_t s, unsigned *flags) {
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_status_attn_tc, sizeof v, 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  e = cudaMemcpyToSymbolAsync(g_status_attn_tc, &zero, sizeof zero, 0,
                              cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  *flags |= v;
  return e;
}

}  // namespace svp
