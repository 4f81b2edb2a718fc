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
// 128-byte-swizzled tiles.  Accumulators live in tensor memory (TMEM).
// A unit is N = 16 or 32 rows of a kv head; beyond 32 rows it is 64 rows
// in two 32-row groups (DUAL), so each K/V tile is read once for all 64,
// and the tensor core takes both groups in one 64-column MMA per k-step
// (the A operand, K or V, is fetched from shared memory once per tile:
// with 32-column MMAs that fetch, not the arithmetic, set the MMA time).
//
// Warp roles (320 threads, one CTA per SM):
//   warps 0-7  softmax and epilogue, as two groups of four warps.  One row
//              group per unit: the groups take alternate tiles (group =
//              tile parity), so one group's shuffles, exponentials and
//              barriers overlap the other's; their states merge by
//              log-sum-exp at the end of a segment.  DUAL: both groups take
//              every tile, one 32-row group each, with S double-buffered;
//              the groups' P (rows 0-31 and 32-63 of one 64-row operand),
//              and at a segment's end their staged outputs, go into the
//              tile's K buffer (read by then), so the ring keeps three
//              stages beside the 64-row Q tile.
//              S is read in the mma-fragment layout (a thread holds four
//              keys of eight rows): row max and sum fold over the four keys
//              in registers, then a short transposing butterfly and a
//              four-warp exchange in shared memory; P goes back to shared
//              memory as bf16 in the MMA's swizzled layout through
//              transposing stmatrix stores.  Interior tiles (every key real
//              and seen by every row) skip per-key masking.  Each group
//              folds its tiles' O into registers (o = o * alpha + O_t).
//   warp 8     producer: block table, 2-D TMA copies of 8 pages' K and V
//              into a 3-stage ring.
//   warp 9     one thread issues tcgen05.mma / tcgen05.commit, event
//              driven: S of a tile as soon as its data and S buffer are
//              free, P V as soon as its P is written, so stages go back to
//              the producer without waiting for later tiles.
// Synchronisation: mbarriers between roles (all waits bounded); named
// barriers inside the softmax warps, where every timeout decision is made
// uniform by an AND-reducing barrier (bar.red.and) before anyone acts on
// it, so no warp can be left waiting at a barrier another warp has left.
// A segment's Q is loaded before the previous segment's epilogue, so the
// tensor core starts on the new segment while the softmax warps write the
// old one out.  Scheduling and the merge of split groups are shared with
// attention.cu (attn_common.cuh).  A timeout raises SVP_DEV_TIMEOUT and every role
// drains what it started before the CTA frees its tensor memory.
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
static_assert(kTilePages == kTilePagesTc, "stream-K items are the kernel's tiles");
constexpr int kHalfBytes = kTileKeys * 128;  // 64 columns x 128 keys, bf16
constexpr int kTileBytes = 2 * kHalfBytes;   // one K (or V) tile: 32 KB
constexpr int kStages = 3;
constexpr int kGroups = 2;                  // softmax groups, by tile parity
constexpr int kGroupThreads = 128;          // four warps: TMEM lanes 0-127
constexpr int kSoftWarps = 4 * kGroups;
constexpr int kProducerWarp = kSoftWarps;
constexpr int kMmaWarp = kSoftWarps + 1;
constexpr int kTcThreads = 32 * (kSoftWarps + 2);
// named barriers (0 is __syncthreads): 1 + g for group g
constexpr int kPageTxBytes = 2 * 2 * kBoxBytes;  // K and V, two boxes each
constexpr int kTcBatchCap = 512;  // sequences per launch (prefix in smem)

// DUAL: a unit holds 2N rows (two row groups of N); both softmax groups
// take every tile, one row group each, so each K/V tile is read once for
// 2N rows.  Its 2N-row Q tile is paid for by keeping P (and a segment's
// staged output) in the stage's K tile, which the tile's S MMAs have
// finished reading by then: no separate P buffers.  Q and P are 2N-row
// K-major operands (group g's rows at g N), so one MMA per k-step serves
// both groups.
template <int N, bool DUAL = false>
struct TcSmem {
  static constexpr int ST = kStages;
  static constexpr int PB = N * kTileKeys * 2;  // one group's P tile (bf16)
  alignas(1024) unsigned char k[ST][kTileBytes];
  alignas(1024) unsigned char v[ST][kTileBytes];
  // Q of a unit's rows: two 64-dim halves, each [rows][128 B] swizzled
  alignas(1024) unsigned char q[(DUAL ? 2 : 1) * N * kD * 2];
  alignas(1024) unsigned char pb[kGroups][DUAL ? 16 : PB];  // P per group
  alignas(16) float red_m[kGroups][4][N];
  alignas(16) float red_l[kGroups][4][N];
  alignas(16) float mu[kGroups][N];        // the max a tile's p was taken at
  alignas(16) float alpha[kGroups][2][N];  // rescale of the state by a tile
  alignas(16) float xs_m[2][N], xs_l[2][N];  // group 1's state per segment
  alignas(16) float f0[N], f1[N];          // combine weights of the groups
  alignas(16) float lse_st[kGroups][N];    // a split partial's LSEs
  uint32_t tbits[kGroups][N];  // draft-tree ancestor bits of the rows
  UnitInfo unit[kUnitRing];
  int stage_mask[ST];  // bit k: page k of the tile was copied
  uint64_t full[ST], empty[ST];
  // S ready: one barrier per group, or per S buffer parity (DUAL: both
  // groups' S MMAs of a tile, one commit)
  uint64_t s_full[2];
  uint64_t p_full[kGroups], o_full[kGroups];
  uint64_t q_full, q_empty;
  uint64_t x_full[2], x_empty[2];  // group 1 -> group 0 state hand-over
  uint64_t stg_free;               // a segment's output left the P buffers
  uint64_t ufull[kUnitRing], uempty[kUnitRing];
  uint64_t drain;
#ifdef SVP_TEST_STALL_AFTER
  uint64_t stall;  // test builds: a barrier nothing arrives on
#endif
  uint32_t tmem_base;
  int abort_flag;
  int prefix[1];  // [batch + 1] item prefix, then [batch] lengths: dynamic
};

template <int N, bool DUAL = false>
constexpr size_t tc_smem_bytes(int batch) {
  return sizeof(TcSmem<N, DUAL>) + sizeof(int) * (2 * (size_t)batch + 1) +
         1024;
}
static_assert(tc_smem_bytes<32>(kTcBatchCap + 1) <= 227 * 1024,
              "shared memory of a 32-row CTA");
static_assert(tc_smem_bytes<16>(kTcBatchCap + 1) <= 227 * 1024,
              "shared memory of a 16-row CTA");
static_assert(tc_smem_bytes<32, true>(kTcBatchCap + 1) <= 227 * 1024,
              "shared memory of a 64-row CTA");
static_assert(TcSmem<32, true>::PB * kGroups <= kTileBytes,
              "the 64-row P operand fits one K tile");
static_assert(32 * kD * 4 * kGroups <= kTileBytes,
              "both groups' fp32 output rows fit one K tile");

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

// Non-blocking test of a phase's completion.
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Named barrier over `count` threads that returns the AND of `ok` over
// them: every participant leaves with the same answer.
__device__ __forceinline__ bool bar_and(int id, int count, bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)ok), "r"(id), "r"(count)
      : "memory");
  return r != 0;
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

// N consecutive 32-bit columns into this thread's TMEM lane.
template <int N>
__device__ __forceinline__ void tmem_st(uint32_t addr, const float (&v)[N]);

template <>
__device__ __forceinline__ void tmem_st<16>(uint32_t addr,
                                            const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,"
      "%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(addr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]),
      "f"(v[6]), "f"(v[7]), "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]),
      "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15])
      : "memory");
}

template <>
__device__ __forceinline__ void tmem_st<32>(uint32_t addr,
                                            const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,"
      "%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,"
      "%26,%27,%28,%29,%30,%31,%32};" ::"r"(addr),
      "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]),
      "f"(v[6]), "f"(v[7]), "f"(v[8]), "f"(v[9]), "f"(v[10]), "f"(v[11]),
      "f"(v[12]), "f"(v[13]), "f"(v[14]), "f"(v[15]), "f"(v[16]), "f"(v[17]),
      "f"(v[18]), "f"(v[19]), "f"(v[20]), "f"(v[21]), "f"(v[22]), "f"(v[23]),
      "f"(v[24]), "f"(v[25]), "f"(v[26]), "f"(v[27]), "f"(v[28]), "f"(v[29]),
      "f"(v[30]), "f"(v[31])
      : "memory");
}

__device__ __forceinline__ void tc_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Byte offset of element (row n, column k) of an [N rows x 128 columns]
// bf16 operand in the K-major 128-byte-swizzled layout: two 64-column
// halves, each [N][128 B], 16-byte chunks XOR-ed with the row mod 8.
template <int N>
__device__ __forceinline__ uint32_t kmajor_off(int n, int k) {
  return (uint32_t)((k >> 6) * (N * 128) + n * 128 +
                    ((((k & 63) >> 3) ^ (n & 7)) << 4) + (k & 7) * 2);
}

// S in the mma-fragment layout: a warp reads its 32 TMEM lanes (keys) as
// two 16-lane halves of 8 J columns (query rows); thread t holds lanes t/4
// and t/4 + 8 of each half, columns 8 i + 2 (t % 4) + {0, 1} of each chunk.
template <int J>
__device__ __forceinline__ void tmem_ld16(uint32_t addr, uint32_t (&r)[4 * J]);

template <>
__device__ __forceinline__ void tmem_ld16<4>(uint32_t addr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,"
      "%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
        "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]),
        "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(addr));
}

template <>
__device__ __forceinline__ void tmem_ld16<2>(uint32_t addr, uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
        "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
      : "r"(addr));
}

// Reduction of a row's values over the 32 keys of a warp: a thread holds
// rows 8 j + 2 (t % 4) + e (already folded over its four keys); lanes of
// equal t % 4 hold the other keys.  A transposing butterfly over lane bits
// 4, 3, 2 leaves lane t with row row_of<J>(t) (J = 2: lanes t and t ^ 4
// share one).
template <int J, bool MAX>
__device__ __forceinline__ float row_reduce(const float (&x)[J][2], int lane) {
  static_assert(J == 2 || J == 4, "16 or 32 rows");
  float v[2 * J];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    v[2 * j] = x[j][0];
    v[2 * j + 1] = x[j][1];
  }
#pragma unroll
  for (int h = J, off = 16; h >= 1; h >>= 1, off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < h; ++i) {
      const float send = upper ? v[i] : v[i + h];
      const float keep = upper ? v[i + h] : v[i];
      const float got = __shfl_xor_sync(kFull, send, off);
      v[i] = MAX ? fmaxf(keep, got) : keep + got;
    }
  }
  if (J == 2) {
    const float got = __shfl_xor_sync(kFull, v[0], 4);
    v[0] = MAX ? fmaxf(v[0], got) : v[0] + got;
  }
  return v[0];
}

template <int J>
__device__ __forceinline__ int row_of(int lane) {
  const int v = J == 4 ? (lane >> 2) & 7 : (lane >> 3) & 3;
  return 8 * (v >> 1) + 2 * (lane & 3) + (v & 1);
}

// Four 8x8 bf16 blocks, stored transposed: this thread's fragment r[i]
// (rows 2 (t % 4) and 2 (t % 4) + 1 of key t / 4) lands in block i, whose
// row t % 8 starts at `addr` of lane 8 i + t % 8.
__device__ __forceinline__ void stmatrix_x4_trans(uint32_t addr,
                                                  const uint32_t (&r)[4]) {
  asm volatile(
      "stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(
          addr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
      : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&h);
}

// K and V caches as 2-D tensors of 16-row pages; Q either as a 3-D tensor
// whose box is a unit's rows (q_unit_box: whole GQA groups of a unit's
// positions, or a whole unit of one position's heads) or as rows of 128
// dims copied one per box.
struct TcMaps {
  CUtensorMap k;
  CUtensorMap v;
  CUtensorMap q;
  int q_unit_box;
};

}  // namespace

// --------------------------------------------------------------------------
// the kernel
// --------------------------------------------------------------------------
template <int N, bool DUAL>
__global__ void __launch_bounds__(kTcThreads, 1)
    paged_attention_tc_kernel(const AttnParams p,
                              const __grid_constant__ TcMaps tm) {
  extern __shared__ unsigned char smem_raw[];
  using Smem = TcSmem<N, DUAL>;
  Smem &sm = *reinterpret_cast<Smem *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int ST = Smem::ST;
  constexpr int UR = DUAL ? 2 * N : N;  // rows of a unit
  // S[group], O[group], X[2] (group 1's o handed to group 0), N columns
  // each; DUAL: S[tile parity] of both groups (2N columns, group g's at
  // g N) at parity 2N, O of both groups at 4N (group g's at (4 + g) N)
  constexpr uint32_t kTmemCols = 6 * N <= 128 ? 128 : 256;
  constexpr uint32_t kIdescS = idesc_bf16(kTileKeys, UR, 0, 0);
  constexpr uint32_t kIdescO = idesc_bf16(kD, UR, 1, 0);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int groups_per_seq = p.num_kv_heads * p.n_rg;

  if (warp == kProducerWarp && lane == 0) {
    prefetch_tensormap(&tm.q);
    prefetch_tensormap(&tm.k);
    prefetch_tensormap(&tm.v);
  }
  if (tid == 0) {
    for (int s = 0; s < ST; ++s) {
      mbar_init(&sm.full[s], 1);
      // DUAL: two commits after the tile's P V (one per group's share),
      // or, for a segment's last tile, each group's arrival once its
      // staged output has been read
      mbar_init(&sm.empty[s], DUAL ? 2 : 1);
    }
    for (int i = 0; i < (int)(sizeof(sm.s_full) / sizeof(uint64_t)); ++i)
      mbar_init(&sm.s_full[i], 1);
    for (int gi = 0; gi < kGroups; ++gi) {
      mbar_init(&sm.p_full[gi], 4);  // the group's warps
      mbar_init(&sm.o_full[gi], 1);
    }
    mbar_init(&sm.q_full, 1);        // the producer's expect_tx + Q copies
    mbar_init(&sm.q_empty, 1);       // the segment's last S MMA completed
    for (int k = 0; k < 2; ++k) {
      mbar_init(&sm.x_full[k], 4);   // group 1's warps
      mbar_init(&sm.x_empty[k], 4);  // group 0's warps
    }
    for (int u = 0; u < kUnitRing; ++u) {
      mbar_init(&sm.ufull[u], 1);
      mbar_init(&sm.uempty[u], 3);   // both softmax groups and the MMA thread
    }
    mbar_init(&sm.stg_free, 1);      // group 0's storing thread
    mbar_init(&sm.drain, 1);
#ifdef SVP_TEST_STALL_AFTER
    mbar_init(&sm.stall, 1);
#endif
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp < kSoftWarps) {
    // Q rows past a segment's valid rows are never copied: keep them zero
    for (int i = tid; i < (int)sizeof(sm.q) / 16; i += kSoftWarps * 32)
      reinterpret_cast<uint4 *>(sm.q)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
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
  tc_fence_before();
  __syncthreads();  // barriers initialised, tensor memory allocated
  tc_fence_after();
  // launched early (programmatic dependent launch): nothing in global
  // memory is touched before the previous kernel on the stream is done --
  // or, right behind the append of the newest positions (p.early), nothing
  // but the pages holding them (the producer waits before the first such
  // tile, the softmax groups before their first output)
  if (!p.early) pdl_wait();
  if (tid == 0) {
    p.desc[blockIdx.x].valid = 0;  // until a split group starts
    pdl_launch_dependents();       // the merge may be scheduled
  }
  const uint32_t tmem = sm.tmem_base;

  if (warp == kProducerWarp) {
    // ======================= producer warp =======================
    // only this warp walks the slices, so it builds the prefix itself
    int *const seqlen = sm.prefix + p.batch + 1;
    const int total_pages = build_prefix(p, sm.prefix, seqlen, groups_per_seq,
                                         lane, &g_status_attn_tc);
    const int n_ctas = working_ctas(total_pages, p.min_pages);
    const int range_begin = slice_begin(blockIdx.x, total_pages, n_ctas);
    const int range_end = blockIdx.x < n_ctas
                              ? slice_begin(blockIdx.x + 1, total_pages, n_ctas)
                              : total_pages;
    int c = 0;   // tiles issued so far
    int us = 0;  // segments published so far
    int q_issued = -1;  // last segment whose Q copies were issued
    bool waited = !p.early;  // the grid-dependency wait is behind us
    bool ok = true;
    int pos = range_begin;
    while (true) {
      const int slot = us % kUnitRing;
      if (lane == 0)
        ok = mbar_wait(&sm.uempty[slot], ((us / kUnitRing) & 1) ^ 1);
      ok = __shfl_sync(kFull, ok, 0) && !sm.abort_flag;
      if (!ok) break;
      const UnitInfo seg =
          pos < range_end
              ? decode_segment(p, sm.prefix, seqlen, groups_per_seq, pos,
                               us == 0, range_end, total_pages, n_ctas)
              : UnitInfo{};
      if (!seg.valid) {
        if (lane == 0) {
          sm.unit[slot].valid = 0;
          mbar_arrive(&sm.ufull[slot]);
        }
        break;
      }
      if (lane == 0) {
        sm.unit[slot] = seg;
        mbar_arrive(&sm.ufull[slot]);
      }
      // Q of the segment's rows, one 128-byte box per half row, once the
      // previous segment's last S MMA has read the old Q; tiles of this
      // segment are issued meanwhile
      bool q_pending = true;
      const int seg_c0 = c;  // the segment's first tile
      auto issue_q = [&]() {
        q_issued = us;
        if (tm.q_unit_box) {
          // the unit's UR rows (row r = position r / group, head r % group
          // from its first row) in one box per 64-dim half; rows past the
          // valid ones hold other rows' queries (or zeros past the tensor)
          // and are never written out.  One copy each instead of one per
          // row: a warp issues bulk copies one at a time
          if (lane == 0) {
            const int gr0 = seg.rg * UR;
            const int y = seg.g * p.group + gr0 % p.group;
            const int z = seg.b * p.q_len + gr0 / p.group;
            mbar_arrive_expect_tx(&sm.q_full, UR * kD * 2);
            tma_load_3d(sm.q, &tm.q, 0, y, z, &sm.q_full);
            tma_load_3d(sm.q + UR * 128, &tm.q, kBoxElems, y, z, &sm.q_full);
          }
          __syncwarp();
        } else {
          const int vr = min(UR, p.rows - seg.rg * UR);
          if (lane == 0) mbar_arrive_expect_tx(&sm.q_full, vr * kD * 2);
          __syncwarp();
          for (int r = lane; r < vr; r += 32) {
            // row r of the unit: 128 B in each 64-dim half of [UR][128 B]
            const int gr = seg.rg * UR + r;
            const int i = gr / p.group, h = seg.g * p.group + gr % p.group;
            const int y = (seg.b * p.q_len + i) * p.num_q_heads + h;
            tma_load_2d(sm.q + r * 128, &tm.q, 0, y, &sm.q_full);
            tma_load_2d(sm.q + UR * 128 + r * 128, &tm.q, kBoxElems, y,
                        &sm.q_full);
          }
        }
        q_pending = false;
      };
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
          if (q_pending) {
            // the stage of tile c last held tile c - ST; if that tile is of
            // this segment its S needs this Q, so the wait for the stage
            // below could only end after it: wait for the old Q's last S
            // (its release is a separate commit, and commits need not
            // arrive in issue order)
            const bool must = c - ST >= seg_c0;
            bool r = false;
            if (lane == 0)
              r = must ? mbar_wait(&sm.q_empty, (us & 1) ^ 1)
                       : mbar_test(&sm.q_empty, (us & 1) ^ 1);
            r = __shfl_sync(kFull, r, 0);
            if (r) {
              issue_q();
            } else if (must) {
              ok = false;
              break;
            }
          }
          // tiles start at multiples of 8 pages of the segment; lane kk < 8
          // copies page t0 + kk, whose entry sits in lane (t0-k0)%32 + kk
          const int npg = min(kTilePages, n_pages - t0);
          if (!waited &&
              (logical_block(seg, seg.page0 + t0 + npg - 1) + 1) * kBlockSize >
                  seg.seq_len - p.q_len) {
            pdl_wait();  // the tile holds some of the appended positions
            waited = true;
          }
          const int k4 = (t0 - k0) >> 5;
          const int src = k4 == 0 ? phys[0] : k4 == 1 ? phys[1]
                        : k4 == 2 ? phys[2] : phys[3];
          const int ph = __shfl_sync(kFull, src, ((t0 - k0) & 31) + (lane & 7));
#ifdef SVP_TEST_STALL_AFTER
          // test builds only: the producer stops after a few tiles and waits
          // on a barrier nothing arrives on, so every role's wait runs out
          if (c == SVP_TEST_STALL_AFTER) {
            bool r = false;
            if (lane == 0) r = mbar_wait(&sm.stall, 0);
            if (!__shfl_sync(kFull, r, 0)) {
              ok = false;
              break;
            }
          }
#endif
          const bool mine = lane < npg;
          const bool good = mine && ph >= 0 && ph < p.num_blocks;
          if (mine && !good) raise_tc(SVP_DEV_BAD_BLOCK_ID);
          const unsigned mask = __ballot_sync(kFull, good) & 0xffu;
          const int s = c % ST;
          if (lane == 0) {
            if (!mbar_wait(&sm.empty[s], ((c / ST) & 1) ^ 1)) {
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
      if (ok && q_pending) {
        if (lane == 0) ok = mbar_wait(&sm.q_empty, (us & 1) ^ 1);
        ok = __shfl_sync(kFull, ok, 0);
        if (ok) issue_q();
      }
      if (!ok) break;
      pos = seg.item0 + (seg.n_pages + p.ppi - 1) / p.ppi;
      ++us;
    }
    if (!ok && lane == 0) {
      // give up: flag it, then wait (bounded) for copies still in flight
      raise_tc(SVP_DEV_TIMEOUT);
      sm.abort_flag = 1;
      for (int k = max(0, c - ST); k < c; ++k)
        (void)mbar_wait_drain(&sm.full[k % ST], (k / ST) & 1);
      if (q_issued >= 0) (void)mbar_wait_drain(&sm.q_full, q_issued & 1);
    }
  } else if (warp == kMmaWarp) {
    // ======================= MMA issuer (event driven) =======================
    if (lane == 0) {
      if constexpr (DUAL) {
        // both groups take every tile, one 2N-column MMA per k-step for
        // both: S(c) (buffer c & 1) once P(c-2) of both was written, one
        // commit; P V(c) once P(c) of both was written, reading the P
        // operand from stage c's K tile, then a commit to each group's O
        // barrier and two to the stage's empty barrier, except on a
        // segment's last tile, whose stage the groups release after their
        // outputs staged there have been read
        bool ok = true;
        int c_s = 0;                 // next tile whose S is issued
        int c_p = 0;                 // next tile whose P V is issued
        int p_obs[2] = {0, 0};       // tiles whose P is known written, by group
        int us = 0;
        int left = 0, tau = 0, cur_pages = 0;
        bool first = false, no_more = false;
        int npg_ring[8];
        bool last_ring[8];
        uint64_t last = globaltimer();
        while (true) {
          bool prog = false;
          if (left == 0 && !no_more &&
              mbar_test(&sm.ufull[us % kUnitRing], (us / kUnitRing) & 1)) {
            const UnitInfo ui = sm.unit[us % kUnitRing];
            mbar_arrive(&sm.uempty[us % kUnitRing]);
            ++us;
            if (!ui.valid) {
              no_more = true;
            } else {
              cur_pages = ui.n_pages;
              left = (ui.n_pages + kTilePages - 1) / kTilePages;
              tau = 0;
              first = true;
            }
            prog = true;
          }
          if (left > 0 && p_obs[0] >= c_s - 1 && p_obs[1] >= c_s - 1 &&
              mbar_test(&sm.full[c_s % ST], (c_s / ST) & 1) &&
              (!first || mbar_test(&sm.q_full, (us - 1) & 1))) {
            tc_fence_after();
            const uint32_t ka = smem_u32(sm.k[c_s % ST]);
            const uint32_t qa = smem_u32(sm.q);
#pragma unroll
            for (int ks = 0; ks < kD / 16; ++ks) {
              const uint64_t a =
                  sw128_desc(ka + (ks >> 2) * kHalfBytes + (ks & 3) * 32, 16, 1024);
              const uint64_t bq =
                  sw128_desc(qa + (ks >> 2) * (UR * 128) + (ks & 3) * 32, 16, 1024);
              tc_mma(tmem + (c_s & 1) * UR, a, bq, kIdescS, ks > 0 ? 1u : 0u);
            }
            // one commit for both groups: when it arrives, K of the tile is
            // no longer read and may take P; S(c + 2) waits for both P(c),
            // so no phase completes twice before both groups have seen it
            tc_commit(&sm.s_full[c_s & 1]);
            npg_ring[c_s & 7] = min(kTilePages, cur_pages - tau * kTilePages);
            last_ring[c_s & 7] = left == 1;
            ++c_s;
            ++tau;
            --left;
            first = false;
            if (left == 0) tc_commit(&sm.q_empty);
            prog = true;
          }
#pragma unroll
          for (int gi = 0; gi < 2; ++gi)
            if (p_obs[gi] < c_s && mbar_test(&sm.p_full[gi], p_obs[gi] & 1)) {
              ++p_obs[gi];
              prog = true;
            }
          if (c_p < p_obs[0] && c_p < p_obs[1]) {
            tc_fence_after();
            const int c = c_p;
            const uint32_t va = smem_u32(sm.v[c % ST]);
            const uint32_t pa = smem_u32(sm.k[c % ST]);
            const int npg = npg_ring[c & 7];
            for (int ks = 0; ks < npg; ++ks) {
              const uint64_t a = sw128_desc(va + ks * 2048, kHalfBytes, 1024);
              const uint64_t bp =
                  sw128_desc(pa + (ks >> 2) * (UR * 128) + (ks & 3) * 32, 16, 1024);
              tc_mma(tmem + 4 * N, a, bp, kIdescO, ks > 0 ? 1u : 0u);
            }
            tc_commit(&sm.o_full[0]);
            tc_commit(&sm.o_full[1]);
            if (!last_ring[c & 7]) {  // one arrival per group's share
              tc_commit(&sm.empty[c % ST]);
              tc_commit(&sm.empty[c % ST]);
            }
            ++c_p;
            prog = true;
          }
          if (no_more && left == 0 && c_p == c_s) break;
          if (prog) {
            last = globaltimer();
          } else if (sm.abort_flag || globaltimer() - last > SVP_WAIT_NS) {
            ok = false;
            break;
          }
        }
        if (!ok) {
          raise_tc(SVP_DEV_TIMEOUT);
          sm.abort_flag = 1;
        }
      } else {
        bool ok = true;
        int c_s = 0;    // next tile whose S is issued
        int c_p = 0;    // next tile whose P V is issued
        int p_obs = 0;  // tiles whose P is known to be written
        int us = 0;     // segments taken from the ring
        int left = 0, tau = 0, cur_pages = 0;
        bool first = false, no_more = false;
        int npg_ring[8];  // pages of tiles c_p .. c_s - 1 (at most 3)
        uint64_t last = globaltimer();
        while (true) {
          bool prog = false;
          // a new segment for the S side
          if (left == 0 && !no_more &&
              mbar_test(&sm.ufull[us % kUnitRing], (us / kUnitRing) & 1)) {
            const UnitInfo ui = sm.unit[us % kUnitRing];
            mbar_arrive(&sm.uempty[us % kUnitRing]);
            ++us;
            if (!ui.valid) {
              no_more = true;
            } else {
              cur_pages = ui.n_pages;
              left = (ui.n_pages + kTilePages - 1) / kTilePages;
              tau = 0;
              first = true;
            }
            prog = true;
          }
          // S^T = K Q^T of tile c_s: its data is in, its group's S buffer was
          // read (P of tile c_s - 2 written), its segment's Q is in
          if (left > 0 && p_obs >= c_s - 1 &&
              mbar_test(&sm.full[c_s % ST], (c_s / ST) & 1) &&
              (!first || mbar_test(&sm.q_full, (us - 1) & 1))) {
            tc_fence_after();
            const int s = c_s % ST, gi = c_s & 1;
            const uint32_t ka = smem_u32(sm.k[s]), qa = smem_u32(sm.q);
  #pragma unroll
            for (int ks = 0; ks < kD / 16; ++ks) {
              // 16 head dims per k-step: 32 B inside the 128-B swizzled rows
              const uint64_t a =
                  sw128_desc(ka + (ks >> 2) * kHalfBytes + (ks & 3) * 32, 16, 1024);
              const uint64_t b =
                  sw128_desc(qa + (ks >> 2) * (N * 128) + (ks & 3) * 32, 16, 1024);
              tc_mma(tmem + gi * N, a, b, kIdescS, ks > 0 ? 1u : 0u);
            }
            tc_commit(&sm.s_full[gi]);
            npg_ring[c_s & 7] = min(kTilePages, cur_pages - tau * kTilePages);
            ++c_s;
            ++tau;
            --left;
            first = false;
            // the segment's last S: its Q may be replaced once this completes
            if (left == 0) tc_commit(&sm.q_empty);
            prog = true;
          }
          if (p_obs < c_s && mbar_test(&sm.p_full[p_obs & 1], (p_obs >> 1) & 1)) {
            ++p_obs;
            prog = true;
          }
          // O_t^T = V^T P^T of tile c_p over its pages (16 keys per k-step);
          // the group read the previous O of this buffer before writing P
          if (c_p < p_obs) {
            tc_fence_after();
            const int s = c_p % ST, gi = c_p & 1;
            const uint32_t va = smem_u32(sm.v[s]), pa = smem_u32(sm.pb[gi]);
            const int npg = npg_ring[c_p & 7];
            for (int ks = 0; ks < npg; ++ks) {
              // V as MN-major A: 64-dim halves kHalfBytes apart (leading byte
              // offset), 8-key groups 1024 B apart (stride byte offset)
              const uint64_t a = sw128_desc(va + ks * 2048, kHalfBytes, 1024);
              const uint64_t b =
                  sw128_desc(pa + (ks >> 2) * (N * 128) + (ks & 3) * 32, 16, 1024);
              tc_mma(tmem + (2 + gi) * N, a, b, kIdescO, ks > 0 ? 1u : 0u);
            }
            tc_commit(&sm.empty[s]);
            tc_commit(&sm.o_full[gi]);
            ++c_p;
            prog = true;
          }
          if (no_more && left == 0 && c_p == c_s) break;
          if (prog) {
            last = globaltimer();
          } else if (sm.abort_flag || globaltimer() - last > SVP_WAIT_NS) {
            ok = false;
            break;
          }
        }
        if (!ok) {
          raise_tc(SVP_DEV_TIMEOUT);
          sm.abort_flag = 1;
        }
      }
      // every MMA issued has completed before tensor memory is freed
      tc_commit(&sm.drain);
      (void)mbar_wait_drain(&sm.drain, 0);
    }
    __syncwarp();
  } else {
    // ======================= softmax groups =======================
    // The two groups run independently: each takes the tiles of its parity
    // in every segment; at a segment's end group 1 parks its state in
    // tensor memory (X[segment & 1]) and moves on, group 0 merges it with
    // its own and writes the segment out.
    const int gi = warp >> 2;          // group: tiles of this parity
    const int gw = warp & 3;           // warp in the group = TMEM lane quadrant
    const int gt = tid & 127;          // head dim of O; row of the stats
    const int gbar = 1 + gi;
    const float qmul = p.qscale > 0.f ? p.qscale : 1.f;
    const uint32_t lane_base = (uint32_t)(gw * 32) << 16;
    const uint32_t tO = tmem + lane_base + (DUAL ? 4 + gi : 2 + gi) * N;
    // phase of this group's t-th tile on its per-group barriers: every tile
    // (DUAL), else every other tile
    auto ph = [](int t) -> uint32_t {
      return DUAL ? (uint32_t)(t & 1) : (uint32_t)((t >> 1) & 1);
    };
    int c0 = 0, us = 0;
    bool ok = true;
    // O of this group's tile t: wait, read, fold into o with alpha(t).
    // Returns a warp-uniform success flag.
    auto fold_o = [&](int t, float (&o)[N]) -> bool {
      const bool got =
          __all_sync(kFull, mbar_wait(&sm.o_full[gi], ph(t)));
      tc_fence_after();
      float ov[N];
      tmem_ld<N>(tO, ov);
      tc_wait_ld();
      const float4 *al =
          reinterpret_cast<const float4 *>(sm.alpha[gi][ph(t)]);
#pragma unroll
      for (int n4 = 0; n4 < N / 4; ++n4) {
        const float4 a = al[n4];
        o[4 * n4 + 0] = fmaf(o[4 * n4 + 0], a.x, ov[4 * n4 + 0]);
        o[4 * n4 + 1] = fmaf(o[4 * n4 + 1], a.y, ov[4 * n4 + 1]);
        o[4 * n4 + 2] = fmaf(o[4 * n4 + 2], a.z, ov[4 * n4 + 2]);
        o[4 * n4 + 3] = fmaf(o[4 * n4 + 3], a.w, ov[4 * n4 + 3]);
      }
      return got;
    };
    while (true) {
      const int slot = us % kUnitRing;
      ok = mbar_wait(&sm.ufull[slot], (us / kUnitRing) & 1);
      ok = bar_and(gbar, kGroupThreads, ok && !sm.abort_flag);
      if (!ok) break;
      const UnitInfo ui = sm.unit[slot];
      if (!ui.valid) break;
      const int b = ui.b, g = ui.g, rg = ui.rg, L = ui.seq_len;
      const int t0 = L - p.q_len;
      // first global row of the group's N rows
      const int row0 = DUAL ? rg * UR + gi * N : rg * N;
      const int vrows = max(0, min(N, p.rows - row0));
      // the rows' draft-tree ancestor bits (all ones without a tree, or
      // past the last query position), read here so that the masked tiles
      // at the segment's end find them in shared memory
      if (gt < N) {
        const int i = (row0 + gt) / p.group;
        sm.tbits[gi][gt] = i < p.q_len ? row_tree_bits(p, b, i) : ~0u;
      }
      named_bar(gbar, kGroupThreads);

      float o[N];
#pragma unroll
      for (int n = 0; n < N; ++n) o[n] = 0.f;
      // running statistics of row gt (thread gt < N of the group)
      float m_run = -INFINITY, l_run = 0.f, alpha_prev = 1.f;
      int prev = -1;  // this group's previous tile in the segment
      const int tiles = (ui.n_pages + kTilePages - 1) / kTilePages;
      for (int tau = DUAL || (c0 & 1) == gi ? 0 : 1; tau < tiles;
           tau += DUAL ? 1 : 2) {
        const int c = c0 + tau;
        const int s = c % ST;
        bool got = mbar_wait(&sm.s_full[DUAL ? (c & 1) : gi], (c >> 1) & 1);
        got = got && mbar_wait(&sm.full[s], (c / ST) & 1);
        tc_fence_after();
        const uint32_t tS =
            tmem + lane_base + (DUAL ? 2 * (c & 1) + gi : gi) * N;
        // S of the tile: key gw 32 + 8 q + lane / 4, query row
        // 8 j + 2 (lane % 4) + e of the group's N rows
        constexpr int J = N / 8;
        float sv[4][J][2];
        {
          uint32_t r0[4 * J], r1[4 * J];
          tmem_ld16<J>(tS, r0);
          tmem_ld16<J>(tS + (16u << 16), r1);
          tc_wait_ld();
#pragma unroll
          for (int j = 0; j < J; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              sv[0][j][e] = __uint_as_float(r0[4 * j + e]);
              sv[1][j][e] = __uint_as_float(r0[4 * j + 2 + e]);
              sv[2][j][e] = __uint_as_float(r1[4 * j + e]);
              sv[3][j][e] = __uint_as_float(r1[4 * j + 2 + e]);
            }
        }

        // S enters the exponent as fma(s, qmul, -mu): with a positive
        // scale the max is taken over raw S and scaled once per row
        // (rounding is monotonic, so that is the max of the scaled S);
        // otherwise S is scaled here and qmul is 1
        if (!(p.qscale > 0.f)) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int j = 0; j < J; ++j) {
              sv[q][j][0] *= p.qscale;
              sv[q][j][1] *= p.qscale;
            }
        }
        // an interior tile: all eight pages copied (a shorter tile's empty
        // slots hold stale keys), no window, every key at or before the
        // first query position (before it, under a draft tree) -- all keys
        // real and seen by every row
        const int npg = min(kTilePages, ui.n_pages - tau * kTilePages);
        const int smask = sm.stage_mask[s];
        const int jlast =
            logical_block(ui, ui.page0 + tau * kTilePages + npg - 1) * kBlockSize +
            kBlockSize - 1;
        const bool interior = p.window == 0 && npg == kTilePages &&
                              smask == (1 << kTilePages) - 1 &&
                              jlast <= t0 - (p.tree_mask ? 1 : 0);
        if (!interior) {
          // this thread's rows: query position and draft-tree ancestor bits
          // (rows past the last query position count as seeing every key)
          int pos[J][2];
          uint32_t tb[J][2];
#pragma unroll
          for (int j = 0; j < J; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int r = 8 * j + 2 * (lane & 3) + e;
              pos[j][e] = t0 + (row0 + r) / p.group;
              tb[j][e] = sm.tbits[gi][r];
            }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int kt = gw * 32 + 8 * q + (lane >> 2);  // key of the tile
            const int kslot = kt >> 4, r = kt & 15;
            const bool loaded = ((smask >> kslot) & 1) != 0;
            const int jk =
                logical_block(ui, ui.page0 + tau * kTilePages + kslot) * kBlockSize + r;
            // visible to some row of the call: holds real data
            const bool in_union = loaded && jk < L &&
                                  (p.window == 0 || jk < p.n_sink || jk > t0 - p.window);
            if (got && kslot < npg && !in_union) {
              // p = 0 here, but 0 * NaN left in unused cache rows is still
              // NaN: the key's four threads clear a quarter of its V row each
#pragma unroll
              for (int c4 = 0; c4 < 4; ++c4) {
                const int idx = (lane & 3) * 4 + c4;
                *reinterpret_cast<uint4 *>(sm.v[s] + (idx >> 3) * kHalfBytes +
                                           kt * 128 + (idx & 7) * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
              }
            }
#pragma unroll
            for (int j = 0; j < J; ++j)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int ps = pos[j][e];
                const bool vis =
                    in_union && jk <= ps &&
                    (p.window == 0 || jk < p.n_sink || jk > ps - p.window) &&
                    (jk < t0 || ((tb[j][e] >> ((jk - t0) & 31)) & 1u) != 0);
                if (!vis) sv[q][j][e] = -INFINITY;
              }
          }
        }

        // ---- row max over the tile's 128 keys ----
        {
          float mx[J][2];
#pragma unroll
          for (int j = 0; j < J; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e)
              mx[j][e] = fmaxf(fmaxf(sv[0][j][e], sv[1][j][e]),
                               fmaxf(sv[2][j][e], sv[3][j][e]));
          const float cm = row_reduce<J, true>(mx, lane);
          if (J == 4 || (lane & 4) == 0) sm.red_m[gi][gw][row_of<J>(lane)] = cm;
        }
        ok = bar_and(gbar, kGroupThreads, ok && got);
        if (!ok) break;
        if (gt < N) {
          const float mt = qmul *
                           fmaxf(fmaxf(sm.red_m[gi][0][gt], sm.red_m[gi][1][gt]),
                                 fmaxf(sm.red_m[gi][2][gt], sm.red_m[gi][3][gt]));
          if (prev >= 0)
            l_run = fmaf(l_run, alpha_prev,
                         (sm.red_l[gi][0][gt] + sm.red_l[gi][1][gt]) +
                             (sm.red_l[gi][2][gt] + sm.red_l[gi][3][gt]));
          const float m_new = fmaxf(m_run, mt);
          const float mu = m_new == -INFINITY ? 0.f : m_new;
          alpha_prev = ex2(m_run - mu);  // 0 while nothing was visible
          m_run = m_new;
          sm.mu[gi][gt] = mu;
          sm.alpha[gi][ph(c)][gt] = alpha_prev;
        }
        named_bar(gbar, kGroupThreads);

        // ---- p = exp2(s - mu) and the row sums ----
        {
          float sm_[J][2];
#pragma unroll
          for (int j = 0; j < J; ++j) {
            const float2 m2 = *reinterpret_cast<const float2 *>(
                &sm.mu[gi][8 * j + 2 * (lane & 3)]);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              sv[q][j][0] = ex2(fmaf(sv[q][j][0], qmul, -m2.x));
              sv[q][j][1] = ex2(fmaf(sv[q][j][1], qmul, -m2.y));
            }
#pragma unroll
            for (int e = 0; e < 2; ++e)
              sm_[j][e] = (sv[0][j][e] + sv[1][j][e]) + (sv[2][j][e] + sv[3][j][e]);
          }
          const float cs = row_reduce<J, false>(sm_, lane);
          if (J == 4 || (lane & 4) == 0) sm.red_l[gi][gw][row_of<J>(lane)] = cs;
        }
        // ---- the previous tile's O leaves the buffer before P is written
        // (the next P V overwrites it; without DUAL that P V has then also
        // finished reading this group's P buffer) ----
        if (prev >= 0) ok = fold_o(prev, o) && ok;
        // group 0 stages the previous segment's output in both P buffers:
        // group 1 writes P again once the TMA engine has read it
        if (!DUAL && gi == 1 && prev < 0 && us > 0)
          ok = __all_sync(kFull, mbar_wait(&sm.stg_free, (us - 1) & 1)) && ok;
        // P as bf16, K-major and swizzled: per 8-row block, four 8x8 blocks
        // (keys gw 32 + 8 i ..) stored transposed.  DUAL: rows gi N .. of
        // the 2N-row operand in the stage's K tile, which the tile's S MMAs
        // have read
        const uint32_t pbase = DUAL ? smem_u32(sm.k[s]) : smem_u32(sm.pb[gi]);
        const int prow0 = DUAL ? gi * N : 0;
#pragma unroll
        for (int j = 0; j < J; ++j) {
          uint32_t fr[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) fr[q] = pack_bf16(sv[q][j][0], sv[q][j][1]);
          stmatrix_x4_trans(
              pbase + kmajor_off<UR>(prow0 + 8 * j + (lane & 7),
                                     gw * 32 + 8 * (lane >> 3)),
              fr);
        }
        fence_proxy_async_smem();  // P and zeroed V rows -> tensor core
        tc_fence_before();         // S and O reads done before they are rewritten
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.p_full[gi]);
        prev = c;
      }
      if (p.early) pdl_wait();  // outputs are written from here on
      // ---- the group's last tile (a warp whose last fold failed skips it;
      // the vote below makes the outcome the group's) ----
      if (ok && prev >= 0) ok = fold_o(prev, o);
      // (also makes the last tile's row sums visible)
      ok = bar_and(gbar, kGroupThreads, ok);
      if (!ok) break;
      if (gt < N && prev >= 0)
        l_run = fmaf(l_run, alpha_prev,
                     (sm.red_l[gi][0][gt] + sm.red_l[gi][1][gt]) +
                         (sm.red_l[gi][2][gt] + sm.red_l[gi][3][gt]));
      const int xk = us & 1;
      const uint32_t tX = tmem + lane_base + (4 + xk) * N;
      if constexpr (DUAL) {
        // ---- epilogue of this group's N rows: no hand-over; staged in
        // the group's half of its last tile's K, where that tile's P was
        // (the tile's P V, which read both groups' P, has completed: the
        // fold above waited for it), and written out by one bulk copy (a
        // partial's rows are consecutive) or one per query position; the
        // stage goes back to the producer once both groups' stores have
        // read it ----
        unsigned char *stg = sm.k[prev % ST] + gi * (kTileBytes / 2);
        const bool single = ui.f == ui.l;
        const size_t pslot = (size_t)(2 * blockIdx.x + ui.slot);
        float *fw = gi == 0 ? sm.f0 : sm.f1;
        if (gt < N) {
          fw[gt] = l_run > 0.f ? 1.f / l_run : 0.f;
          const float lse2 = l_run > 0.f ? m_run + log2f(l_run) : -INFINITY;
          if (single) {
            if (gt < vrows) {
              const int gr = row0 + gt;
              const int i = gr / p.group, h = g * p.group + gr % p.group;
              p.lse[((size_t)b * p.q_len + i) * p.num_q_heads + h] = lse2 * kLn2;
            }
          } else {
            sm.lse_st[gi][gt] = lse2;
          }
        }
        named_bar(gbar, kGroupThreads);
        if (single) {
          __nv_bfloat16 *stg16 = reinterpret_cast<__nv_bfloat16 *>(stg);
#pragma unroll
          for (int n = 0; n < N; ++n)
            stg16[n * kD + gt] = __float2bfloat16_rn(o[n] * fw[n]);
          fence_proxy_async_smem();
          named_bar(gbar, kGroupThreads);
          if (gt == 0) {
            for (int n = 0; n < vrows;) {
              const int gr = row0 + n, i = gr / p.group;
              const int n_end = min(vrows, (i + 1) * p.group - row0);
              const int h = g * p.group + gr % p.group;
              bulk_s2g(static_cast<uint16_t *>(p.out) +
                           (((size_t)b * p.q_len + i) * p.num_q_heads + h) * kD,
                       stg16 + n * kD, (uint32_t)(n_end - n) * kD * 2);
              n = n_end;
            }
            bulk_commit();
            bulk_wait_read();
          }
        } else {
          // fp32 rows [N][128]: the group's rows of this CTA's partial slot
          float *stg32 = reinterpret_cast<float *>(stg);
#pragma unroll
          for (int n = 0; n < N; ++n) stg32[n * kD + gt] = o[n] * fw[n];
          fence_proxy_async_smem();
          named_bar(gbar, kGroupThreads);
          if (gt == 0) {
            bulk_s2g(p.part_o + (pslot * UR + gi * N) * kD, stg32, N * kD * 4);
            bulk_s2g(p.part_lse + pslot * UR + gi * N, sm.lse_st[gi], N * 4);
            bulk_commit();
            bulk_wait_read();
            if (gi == 0) record_split(p, ui, blockIdx.x);
          }
        }
        // fw and the staging area are rewritten only after this barrier;
        // then the last tile's stage may be refilled
        named_bar(gbar, kGroupThreads);
        if (gt == 0) mbar_arrive(&sm.empty[prev % ST]);
      } else if (gi == 1) {
        // ---- hand the state to group 0 (its copy of segment us - 2 must
        // have been taken) and go on with the next segment ----
        bool got = us < 2 || mbar_wait(&sm.x_empty[xk], ((us >> 1) - 1) & 1);
        ok = bar_and(gbar, kGroupThreads, got);
        if (!ok) break;
        tc_fence_after();
        tmem_st<N>(tX, o);
        if (gt < N) { sm.xs_m[xk][gt] = m_run; sm.xs_l[xk][gt] = l_run; }
        tc_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.x_full[xk]);
      } else {
        // ---- epilogue (group 0): merge the two groups' states; a group
        // owned by one CTA is finished here, else a partial goes to this
        // CTA's first- or last-segment slot ----
        bool got = mbar_wait(&sm.x_full[xk], (us >> 1) & 1);
        ok = bar_and(gbar, kGroupThreads, got);
        if (!ok) break;
        tc_fence_after();
        float o1[N];
        tmem_ld<N>(tX, o1);
        tc_wait_ld();
        const bool single = ui.f == ui.l;
        const size_t pslot = (size_t)(2 * blockIdx.x + ui.slot);
        if (gt < N) {
          const float m1 = sm.xs_m[xk][gt], l1 = sm.xs_l[xk][gt];
          const float M = fmaxf(m_run, m1);
          const float mr = M == -INFINITY ? 0.f : M;
          const float w0 = ex2(m_run - mr), w1 = ex2(m1 - mr);
          const float lt = w0 * l_run + w1 * l1;
          const float inv = lt > 0.f ? 1.f / lt : 0.f;
          sm.f0[gt] = w0 * inv;
          sm.f1[gt] = w1 * inv;
          const float lse2 = lt > 0.f ? mr + log2f(lt) : -INFINITY;
          if (single) {
            if (gt < vrows) {
              const int gr = row0 + gt;
              const int i = gr / p.group, h = g * p.group + gr % p.group;
              p.lse[((size_t)b * p.q_len + i) * p.num_q_heads + h] = lse2 * kLn2;
            }
          } else {
            sm.lse_st[0][gt] = lse2;
          }
        }
        // group 1's state is read: its slot may be reused
        tc_fence_before();
        named_bar(gbar, kGroupThreads);
        if (lane == 0) mbar_arrive(&sm.x_empty[xk]);
        // ---- the rows go out through the TMA engine, staged in the P
        // buffers (every P V of the segment is done; group 1 writes P again
        // after stg_free): plain stores would queue behind the KV stream of
        // all SMs and stall this group for microseconds ----
        float *stg32 = reinterpret_cast<float *>(&sm.pb[0][0]);  // [N][128]
        __nv_bfloat16 *stg16 = reinterpret_cast<__nv_bfloat16 *>(&sm.pb[0][0]);
#pragma unroll
        for (int n = 0; n < N; ++n) {
          const float val = o[n] * sm.f0[n] + o1[n] * sm.f1[n];
          if (single)
            stg16[n * kD + gt] = __float2bfloat16_rn(val);
          else
            stg32[n * kD + gt] = val;
        }
        fence_proxy_async_smem();
        named_bar(gbar, kGroupThreads);
        if (gt == 0) {
          if (single) {
            // one copy per query position: its rows are consecutive heads
            for (int n = 0; n < vrows;) {
              const int gr = row0 + n, i = gr / p.group;
              const int n_end = min(vrows, (i + 1) * p.group - row0);
              const int h = g * p.group + gr % p.group;
              bulk_s2g(static_cast<uint16_t *>(p.out) +
                           (((size_t)b * p.q_len + i) * p.num_q_heads + h) * kD,
                       stg16 + n * kD, (uint32_t)(n_end - n) * kD * 2);
              n = n_end;
            }
          } else {
            bulk_s2g(p.part_o + pslot * N * kD, stg32, N * kD * 4);
            bulk_s2g(p.part_lse + pslot * N, sm.lse_st[0], N * 4);
            record_split(p, ui, blockIdx.x);
          }
          bulk_commit();
          bulk_wait_read();  // the staging area may be written again
          mbar_arrive(&sm.stg_free);
        }
        // f0 / f1 / the staging area are rewritten only after this barrier
        named_bar(gbar, kGroupThreads);
      }
      if (gt == 0) mbar_arrive(&sm.uempty[slot]);
      c0 += tiles;
      ++us;
    }
    if (!ok && gt == 0) {
      raise_tc(SVP_DEV_TIMEOUT);
      sm.abort_flag = 1;
    }
    // the output stores have landed
    if (DUAL ? gt < N : gi == 0 && gt == 0) bulk_wait();
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

template <int N, bool DUAL>
static int prepare_tc(int batch) {
  const size_t smem = tc_smem_bytes<N, DUAL>((int)tc_batch_bucket(batch));
  auto kern = paged_attention_tc_kernel<N, DUAL>;
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

template <int N, bool DUAL>
static cudaError_t launch_tc(const AttnParams &p, int grid, cudaStream_t st) {
  if (prepare_tc<N, DUAL>(p.batch) < 0) return cudaErrorInvalidValue;
  const size_t smem = tc_smem_bytes<N, DUAL>((int)tc_batch_bucket(p.batch));
  TcMaps tm;
  memset(&tm, 0, sizeof tm);
  // a unit's rows as one box: whole GQA groups of UR / group positions, or
  // UR heads of one position (every unit then starts on a box boundary)
  constexpr int UR = DUAL ? 2 * N : N;
  const long long positions = (long long)p.batch * p.q_len;
  int bh = 0, bp = 0;
  if (p.group <= UR && UR % p.group == 0) {
    bh = p.group;
    bp = UR / p.group;
  } else if (p.group > UR && p.group % UR == 0) {
    bh = UR;
    bp = 1;
  }
  tm.q_unit_box = bh > 0 && bp <= positions;
  if (!cached_map(&tm.k, 0, p.k_cache, p.num_blocks, p.num_kv_heads, kD) ||
      !cached_map(&tm.v, 0, p.v_cache, p.num_blocks, p.num_kv_heads, kD) ||
      !(tm.q_unit_box
            ? cached_map(&tm.q, 2, p.q, positions, p.num_q_heads, kD,
                         bh * 65536 + bp)
            : cached_map(&tm.q, 1, p.q, positions * p.num_q_heads, 0, kD)))
    return cudaErrorInvalidValue;
  return launch_pdl(paged_attention_tc_kernel<N, DUAL>, (unsigned)grid,
                    (unsigned)kTcThreads, smem, st, p, tm);
}

int tc_batch_cap() { return kTcBatchCap; }

int attention_tc_ctas_per_sm(int rb, int batch) {
  const int n = rb == 16   ? prepare_tc<16, false>(batch)
                : rb == 32 ? prepare_tc<32, false>(batch)
                           : prepare_tc<32, true>(batch);
  return n > 0 ? n : 1;
}

cudaError_t launch_attention_tc(const AttnParams &p, int grid,
                                cudaStream_t stream) {
  if (p.head_dim != kD || (p.rb != 16 && p.rb != 32 && p.rb != 64) ||
      p.batch > kTcBatchCap)
    return cudaErrorInvalidValue;
  return p.rb == 16   ? launch_tc<16, false>(p, grid, stream)
         : p.rb == 32 ? launch_tc<32, false>(p, grid, stream)
                      : launch_tc<32, true>(p, grid, stream);
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
