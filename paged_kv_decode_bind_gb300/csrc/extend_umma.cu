// Paged extend (prefill) attention on the fifth-generation tensor cores:
// tcgen05.mma with both contractions' accumulators in tensor memory (TMEM).
// Same arguments, units, outputs and error rules as the warp-level kernel in
// extend_mma.cu (the engine keeps the prefill step's qo_indptr in its
// workspace: workspace.py page, bullet 19), which still serves the layouts
// this one does not carry: flat token indices and page sizes that are not a
// multiple of 16.
//
// A CTA owns 128 query rows of one (request, KV head): 128 / G new tokens x
// the G query heads of the group, row r = (token r / G, head r % G), so a key
// tile is read once for the whole group.  Per 128-key tile:
//   S = Q K^T   tcgen05.mma M = 128, N = 128, K = D in steps of 16.  Q is the
//               A operand from TMEM (D / 2 columns of bf16 pairs a row, stored
//               by the softmax warps), which leaves shared memory to a
//               3-stage K ring; the tile's K sits K-major in shared memory
//               with the 128-byte swizzle ([64-column half][rows][128 B]); S
//               lands in one of two 128-column TMEM buffers, so the next
//               tile's product runs while this tile's softmax reads its own.
//               (N = 128: measured, an N = 64 MMA runs at about half the
//               tensor rate.)
//   softmax     two threads per row, 64 keys each: a thread loads its half
//               row of S from TMEM (tcgen05.ld), applies the causal mask,
//               swaps its partial maximum with the other half's thread
//               through shared memory, keeps the running max and sum in fp32
//               (exp2) and writes the weights P back into the same TMEM
//               buffer as bf16 high and low parts, P = P_hi + P_lo to ~2^-17
//               (pairs of keys per 32-bit column).
//   O += P V    tcgen05.mma M = 128, N = D, K = 128 keys in steps of 16 with
//               P_hi and P_lo each as the A operand from TMEM and V read from
//               shared memory as an MN-major operand (the tile's V rows,
//               [half][key][128 B], are rows of 64 dims).  O stays in TMEM
//               for the unit's whole key range.
// A row's reference maximum is raised, and its O row rescaled through
// tcgen05.ld / st, only when a tile's maximum exceeds it by more than 2^8;
// the weights exp2(s - m) then stay below 256 and the sum and O use the same
// reference, so the result is unchanged.
//
// Warps: 0 and 10 issue the tensor-map boxes of each tile's K and V (per
// 16-token page piece one box per 64-column half) into 3-stage K and V
// rings; 1 issues every tile's Q K^T and 11 every P V (each from one
// lane chosen by elect.sync while the whole warp runs the loop), tracking
// their completion with tcgen05.commit on mbarriers; 2-9 load Q, run the
// softmax (two warps per TMEM lane quarter, 64 keys of a tile each) and write
// the outputs.  Every wait is bounded (~1 s) and raises PKV_DEVERR_TIMEOUT;
// the MMAs in flight are drained before the TMEM is freed.
#include <cuda.h>

#include <cstring>

#include "extend_common.cuh"

namespace pkv {

namespace {

constexpr int kUM = 128;          // query rows per CTA (TMEM lanes)
constexpr int kUN = 128;          // keys per tile (N of Q K^T: the MMA's full rate)
constexpr int kUKStages = 3;      // K ring: a tile's K is free once its Q K^T is done
constexpr int kUVStages = 3;      // V ring: free once the tile's P V is done
constexpr int kUSBufs = 2;        // S / P buffers in TMEM
constexpr int kUSoftWarps = 8;    // two per TMEM lane quarter, 64 keys of a tile each
// warps: K loader, Q K^T issuer, softmax, V loader, P V issuer
constexpr int kUThreads = (4 + kUSoftWarps) * 32;
constexpr int kUVWarp = 2 + kUSoftWarps;
constexpr int kUPVWarp = 3 + kUSoftWarps;
constexpr int kUTmemCols = 512;   // two S buffers of 128 columns, O of D <= 128, Q of D / 2
constexpr int kUOCol = kUSBufs * kUN;  // O's first column
constexpr int kUQCol = kUOCol + 128;   // Q's first column: bf16 pairs, D / 2 columns
constexpr float kURescale = 8.f;  // raise a row's reference max only past this (log2)
constexpr int kUSortMax = 256;    // (query block, split, request) triples ordered by cost

template <int D>
struct UCfg {
  static constexpr int HALVES = D / 64;
  static constexpr int KSTEPS = D / 16;
  static constexpr int KVHALF = kUN * 128;  // one half of a tile's K (or V)
  static constexpr int KBYTES = HALVES * KVHALF;  // a tile's K (or V)
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + kUKStages * KBYTES;
  static constexpr int SMEM = OFF_V + kUVStages * KBYTES + 1024;  // + alignment slack
  static constexpr uint32_t PIECE_TX = HALVES * 16 * 128;  // K (or V) of 16 tokens
  static_assert(D == 64 || D == 128, "one or two 64-column halves");
  static_assert(D <= kUQCol - kUOCol, "O fits below Q");
  static_assert(kUQCol + D / 2 <= kUTmemCols, "Q fits the allocation");
  static_assert(SMEM + 8192 <= 227 * 1024, "shared memory of one CTA");
};

// Shared-memory matrix descriptor of tcgen05.mma: start address, leading and
// stride byte offsets (16-byte units), the descriptor version bit (46) and
// the 128-byte swizzle (2 at bit 61).  K-major operands: rows 128 B apart,
// 8-row groups SBO apart, LBO unused; MN-major: LBO between 64-element
// blocks of the MN dimension, SBO between groups of 8 K rows.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of kind::f16: fp32 accumulator (bits 4-5), bf16 A
// (7-9) and B (10-12), A K-major, B K-major or MN-major (bit 16), N / 8
// (17-22), M / 16 (24-28).
__host__ __device__ constexpr uint32_t umma_idesc(int M, int N, int b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn_major << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// The MMA warp runs its loop with all 32 lanes (so its operands stay
// warp-uniform) and one lane, chosen by elect.sync, issues each instruction.
// Measured: an MMA stream issued from a lone divergent lane ran 3x slower
// while other warps of its SM sub-partition kept the issue slots busy (the
// softmax warps here); issued this way it ran within 2 % of its rate alone.
// Both products take their A operand (M x 16, bf16 pairs per 32-bit column)
// from TMEM and B from a shared-memory descriptor.
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                        uint32_t idesc, int accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive (once) on the mbarrier when every MMA issued so far is done.  The
// elected lane is the one that issued them (the warp is converged: the
// lowest lane every time), as the commit tracks its own thread's MMAs.
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 32 consecutive 32-bit TMEM columns of this thread's lane (warp-collective).
__device__ __forceinline__ void tmem_ld32(uint32_t (&r)[32], uint32_t taddr) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 2^x with the SFU's ex2.approx (relative error ~2^-22, far below the
// weights' bf16 high + low rounding); 2^-inf = 0.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// mbarrier phase wait that suspends the thread in hardware (up to the hint)
// instead of spinning, bounded like mbar_wait_bounded: false after ~1 s.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity), "r"(1000000u)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait_sleep(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity)) return true;
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
}

// Blackwell's paired fp32 arithmetic: two lanes of a 64-bit register pair
// per instruction (x in the low word).
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  return ((uint64_t)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ float f2_lo(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f2_hi(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
// max of three (one instruction on this architecture)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t x, uint32_t y, uint32_t z,
                                             uint32_t w) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(x), "r"(y), "r"(z),
               "r"(w)
               : "memory");
}

// One tensor-map box, issued by one lane chosen by elect.sync; the whole
// warp executes it with the same (warp-uniform) operands.  Measured: boxes
// issued this way cost about a third of the per-lane issue (each lane its own
// box), whose issue also slowed 3x while other warps of the sub-partition
// were busy.
__device__ __forceinline__ void tma_box(uint32_t dst, const CUtensorMap *tm, int c1, int c2,
                                        int c3, uint64_t *bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], "
      "[%1, {%2, %3, %4, %5}], [%6];\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ int unit_tiles(const XUnit &x) {
  return x.k1 > x.k0 ? (x.k1 - x.k0 + kUN - 1) / kUN : 0;
}

template <int D, int G>
__global__ void __launch_bounds__(kUThreads, 1)
    extend_umma_kernel(const __grid_constant__ XArgs a, const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv) {
  // Anything read here may come from the previous kernel on the stream
  // (programmatic dependent launch): wait for it, then let the next start.
  // With PKV_FLAG_PLAN_EARLY the metadata, the page table and the cached
  // tokens' K/V are older than that kernel, so the CTA orders its units and
  // its loaders fetch the cached tiles first; the loaders wait before a tile
  // that holds new tokens, the softmax warps before reading q or writing.
  const bool early = (a.flags & PKV_FLAG_PLAN_EARLY) != 0;
  if (!early) pdl_wait();
  pdl_trigger();
  using C = UCfg<D>;
  constexpr int TQ = kUM / G;  // new tokens per CTA
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t k_full[kUKStages], k_empty[kUKStages];
  __shared__ __align__(8) uint64_t v_full[kUVStages], v_empty[kUVStages];
  __shared__ __align__(8) uint64_t s_full[kUSBufs], buf_free[kUSBufs];
  // p_full rotates over the S buffers: the Q K^T of the next tiles may
  // already be done when the P V warp looks for tile kk's P, so the softmax
  // could publish theirs too; one barrier would then have passed the phase
  // looked for
  __shared__ __align__(8) uint64_t q_full, p_full[kUSBufs], drain[2];
  __shared__ __align__(8) uint64_t xbar[4];  // per lane quarter: its two softmax warps
  // Bad page bits of the CTA's i-th unit in s_ubad[i % 4], written by the V
  // loader before it publishes each of the unit's tiles (set by the first,
  // OR-ed by the rest); the softmax reads them once the unit's last V tile
  // has landed, and the loader is then at most three tiles, so three units,
  // ahead of it.  (A K
  // stage is refilled as soon as its Q K^T is done, possibly before the
  // softmax of its tile has started, so the K side carries no flags.)
  __shared__ int s_ubad[4];
  __shared__ float s_xmax[2][2][kUM];  // [tile parity][key half][row]: partial row maxima
  __shared__ float s_xsum[2][kUM];     // [key half][row]: partial row sums, at the end
  __shared__ int s_cost[kUSortMax], s_order[kUSortMax];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  uint8_t *smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_addr(smem);
  const pkv_workspace &ws = a.ws;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Hq = ws.n_q_heads;
  const int jmax = (a.max_qo_len + TQ - 1) / TQ;
  const int units = jmax * a.S * a.batch * ws.n_kv_heads;
  if (tid == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmk) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(&tmv) : "memory");
    for (int s = 0; s < kUKStages; ++s) {
      mbar_init(&k_full[s], 1);   // the K loader's expect-tx arrival
      mbar_init(&k_empty[s], 1);  // commit after the tile's Q K^T
    }
    for (int s = 0; s < kUVStages; ++s) {
      mbar_init(&v_full[s], 1);   // the V loader's expect-tx arrival
      mbar_init(&v_empty[s], 1);  // commit after the tile's P V
    }
    for (int i = 0; i < kUSBufs; ++i) {
      mbar_init(&s_full[i], 1);    // commit after the tile's Q K^T
      // commit after the tile's P V (P read from the buffer, O holds the tile);
      // the softmax waits here for O too.  One barrier per buffer: waiting
      // on the P V of tile kk, the barrier's previous phase (tile kk - 2) is
      // complete and its next (tile kk + 2) needs a P not yet written, so a
      // parity wait cannot pass early, as it could on a single barrier two
      // phases behind once Q K^T runs ahead.
      mbar_init(&buf_free[i], 1);
    }
    mbar_init(&q_full, kUSoftWarps);  // the softmax warps have written Q
    for (int i = 0; i < kUSBufs; ++i) mbar_init(&p_full[i], kUSoftWarps);  // ... and P
    mbar_init(&drain[0], 1);
    mbar_init(&drain[1], 1);
    for (int i = 0; i < 4; ++i) {
      mbar_init(&xbar[i], 2);
      s_ubad[i] = 0;
    }
    s_abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(&s_tmem)),
                 "r"(kUTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // Work order.  Units are (query block j, split c, request b, KV head g);
  // the heads of a (j, c, b) triple cost the same.  With at most kUSortMax
  // triples every CTA ranks them by tile count (descending, ties by index),
  // then takes positions in snake order over that list: i-th round position
  // i * grid + blockIdx.x, every other round reversed, so the CTA with the
  // costliest unit takes the cheapest of the next round.
  const int n3 = jmax * a.S * a.batch, hkv = ws.n_kv_heads;
  const bool ranked = n3 <= kUSortMax;
  if (ranked) {
    for (int t = tid; t < n3; t += kUThreads) {
      const XUnit x = xunit(a, t * hkv, TQ, jmax);
      s_cost[t] = x.live ? unit_tiles(x) : 0;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (ranked) {
    for (int t = tid; t < n3; t += kUThreads) {
      const int ct = s_cost[t];
      int rank = 0;
      for (int o = 0; o < n3; ++o) {
        const int co = s_cost[o];
        rank += (co > ct) || (co == ct && o < t);
      }
      s_order[rank] = t;
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  // the CTA's i-th unit, or -1 past the last
  auto unit_of = [&](int i) -> int {
    const long long pos = (i & 1) ? (long long)(i + 1) * gridDim.x - 1 - blockIdx.x
                                  : (long long)i * gridDim.x + blockIdx.x;
    if (pos >= units) return -1;
    const int t3 = ranked ? s_order[pos / hkv] : (int)(pos / hkv);
    return t3 * hkv + (int)(pos % hkv);
  };

  // A bounded wait; one that runs out stops the whole CTA.
  auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
    if (mbar_try_wait(bar, parity)) return true;
    if (s_abort) return false;
    if (mbar_wait_sleep(bar, parity)) return true;
    s_abort = 1;
    atomicOr(ws.err, PKV_DEVERR_TIMEOUT);
    return false;
  };

  if (warp == 0 || warp == kUVWarp) {
    // ------------------------------------------------------- loaders ----
    // Warp 0 loads each tile's K into the K ring, the last warp its V into
    // the V ring.  Lane j & 7 looks up the slot of piece j of the tile's
    // eight 16-token pieces; the warp then issues the boxes (piece x 64-column
    // half).  A bad page id loads the in-range slot 0 instead (both loaders
    // raise its error bit) and flags the V stage (its unit is written empty).
    const bool isv = warp == kUVWarp;
    const int nst = isv ? kUVStages : kUKStages;
    uint64_t *fullb = isv ? v_full : k_full;
    uint64_t *emptyb = isv ? v_empty : k_empty;
    const CUtensorMap *tm = isv ? &tmv : &tmk;
    const uint32_t ring = sbase + (isv ? C::OFF_V : C::OFF_K);
    Plan pl;
    pl.set_pages(ws);
    const int j = lane & 7;
    int k = 0;
    bool aborted = false, waited = !early;
    for (int ui = 0, u; !aborted && (u = unit_of(ui)) >= 0; ++ui) {
      const XUnit x = xunit(a, u, TQ, jmax);
      if (!x.live) continue;
      // keys below this are the request's cached tokens (every key of the
      // context when the query rows are not tokens of it)
      const int cached = (a.flags & PKV_FLAG_EXTEND_FULL) ? x.L : x.L - x.n;
      const int rrow = ws.req_pool_indices[x.b];
      const bool row_ok = rrow >= 0 && rrow < ws.max_reqs;
      const long long base = row_ok ? (long long)rrow * ws.max_pages_per_req : 0;
      auto raw_at = [&](int t) {
        return (t >= x.k1 || !row_ok) ? -1 : ws.page_table[base + pl.page_of(t)];
      };
      const int ntiles = unit_tiles(x);
      int raw = raw_at(x.k0 + 16 * j);
      for (int tile = 0; tile < ntiles; ++tile, ++k) {
        const int s = k % nst, r = k / nst;
        // the decision is the warp's (the boxes below are issued by all lanes)
        if (!__all_sync(0xffffffffu, !((r > 0 && !wait(&emptyb[s], (r - 1) & 1)) || s_abort))) {
          aborted = true;
          break;
        }
        const int t0 = x.k0 + tile * kUN;
        if (!waited && min(t0 + kUN, x.k1) > cached) {
          pdl_wait();  // the tile holds new tokens: their rows may be the previous kernel's
          waited = true;
        }
        const int np = min(kUN / 16, (x.k1 - t0 + 15) / 16);
        int kind = 0, slot0 = 0;
        if (j < np) {
          const long long s0 = slot_from_raw(ws, pl, raw, t0 + 16 * j, kind);
          if (!kind) slot0 = (int)s0;
        }
        const int nx = raw_at(t0 + kUN + 16 * j);  // the next tile's, while these issue
        const int bad = __reduce_or_sync(0xffffffffu, kind);
        if (lane == 0) {
          // the unit's first tile sets the bits, later tiles add to them
          if (isv && tile == 0) s_ubad[ui & 3] = bad;
          else if (isv && bad) atomicOr(&s_ubad[ui & 3], bad);
          if (bad) atomicOr(ws.err, bad);
        }
        __syncwarp();
        // the boxes, one after another from the whole warp: piece pj's slot
        // comes from lane pj
        for (int pj = 0; pj < np; ++pj) {
          const int sl = __shfl_sync(0xffffffffu, slot0, pj);
#pragma unroll
          for (int hh = 0; hh < C::HALVES; ++hh)
            tma_box(ring + s * C::KBYTES + hh * C::KVHALF + pj * 2048, tm,
                    a.layer * ws.pool_slots + sl, hh, x.g, &fullb[s]);
        }
        if (lane == 0) mbar_arrive_expect_tx(&fullb[s], np * C::PIECE_TX);
        raw = nx;
      }
    }
    if (aborted) {
      // the last (up to nst) tiles issued may still be landing
      for (int kk = max(0, k - nst); kk < k; ++kk) mbar_wait_bounded(&fullb[kk % nst], (kk / nst) & 1);
    }
  } else if (warp == 1 || warp == kUPVWarp) {
    // ------------------------------------------------------------ MMA ----
    // Two issuing warps, so that neither kind of product waits behind the
    // other's barriers: warp 1 issues every tile's S = Q K^T as soon as its K
    // has landed and its S / P buffer is free (the P V of the tile two
    // before is done); the P V warp issues O += P V as soon as the softmax
    // has written the tile's P and its V has landed.  The tensor pipe takes
    // both streams; each warp's commits track its own products.
    const bool pv = warp == kUPVWarp;
    // a wait that fails for any lane stops the warp
    auto wwait = [&](uint64_t *bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, wait(bar, parity));
    };
    constexpr uint32_t kIdS = umma_idesc(kUM, kUN, 0);  // S = Q K^T: both K-major
    constexpr uint32_t kIdO = umma_idesc(kUM, D, 1);    // O += P V: V MN-major
    // descriptors of stage 0's K and V; every other shared-memory operand is
    // one of these plus a byte offset (in 16-byte units, inside the start
    // field)
    const uint64_t dk = umma_desc(sbase + C::OFF_K, 16, 1024);
    const uint64_t dv = umma_desc(sbase + C::OFF_V, C::KVHALF, 1024);
    int k = 0, ul = 0;
    bool dead = false;
    for (int ui = 0, u; !dead && (u = unit_of(ui)) >= 0; ++ui) {
      const XUnit x = xunit(a, u, TQ, jmax);
      if (!x.live) continue;
      const int T = unit_tiles(x);
      if (T == 0) continue;
      if (!pv) {
        if (!wwait(&q_full, ul & 1)) break;
        tc_fence_after();
      }
      for (int t = 0; t < T && !dead; ++t) {
        const int kk = k + t, b = kk % kUSBufs;
        if (!pv) {
          const int s = kk % kUKStages;
          if (!wwait(&k_full[s], (kk / kUKStages) & 1) ||
              (kk >= kUSBufs && !wwait(&buf_free[b], ((kk / kUSBufs) - 1) & 1))) {
            dead = true;
            break;
          }
          tc_fence_after();
          const uint64_t ks0 = (uint64_t)((s * C::KBYTES) >> 4);
#pragma unroll
          for (int ks = 0; ks < C::KSTEPS; ++ks) {
            // k-step ks: Q's columns 8 ks .. 8 ks + 7 (16 dims as bf16 pairs);
            // K's half ks / 4, 32 bytes further per step inside the rows
            const uint64_t ko = (uint64_t)(((ks >> 2) * C::KVHALF + (ks & 3) * 32) >> 4);
            umma_ts(tmem + b * kUN, tmem + kUQCol + ks * 8, dk + ks0 + ko, kIdS, ks > 0);
          }
          umma_commit(&s_full[b]);
          umma_commit(&k_empty[s]);
        } else {
          const int s = kk % kUVStages;
          if (!wwait(&p_full[b], (kk / kUSBufs) & 1) || !wwait(&v_full[s], (kk / kUVStages) & 1)) {
            dead = true;
            break;
          }
          tc_fence_after();
          const uint64_t vs0 = (uint64_t)((s * C::KBYTES) >> 4);
          const uint32_t pb = tmem + b * kUN;  // P_hi in the buffer's first 64 columns
#pragma unroll
          for (int ks = 0; ks < kUN / 16; ++ks) {
            // 16 keys per step: 16 V rows (2048 B) further, 8 P columns
            const uint64_t bd = dv + vs0 + (uint64_t)((ks * 2048) >> 4);
            umma_ts(tmem + kUOCol, pb + ks * 8, bd, kIdO, t > 0 || ks > 0);
            umma_ts(tmem + kUOCol, pb + kUN / 2 + ks * 8, bd, kIdO, 1);
          }
          umma_commit(&buf_free[b]);
          umma_commit(&v_empty[s]);
        }
      }
      k += T;
      ++ul;
    }
    // every MMA this warp issued is done before the TMEM is freed
    umma_commit(&drain[pv]);
    mbar_wait_bounded(&drain[pv], 0);
    __syncwarp();
  } else {
    // -------------------------------------------------------- softmax ----
    // Warp w owns TMEM lane quarter w % 4 (rows 32 (w % 4) .. + 31) and key
    // half hf of every tile (columns 64 hf .. + 63 of S, 32 hf .. of P_hi and
    // P_lo) and half hf of O's columns; the two threads of a row swap their
    // partial maxima (and, at the end, sums) through shared memory, meeting
    // on the quarter's mbarrier (a bounded wait, like every other).
    const int wq = warp & 3, hf = (warp - 2) >> 2;
    const int row = 32 * wq + lane;
    const uint32_t trow = tmem + ((uint32_t)(32 * wq) << 16);
    const float qk_scale = a.scale * kLog2e;
    const bool pos_scale = qk_scale > 0.f;
    const bool full_mode = (a.flags & PKV_FLAG_EXTEND_FULL) != 0;
    if (early) pdl_wait();  // q and the outputs
    const bool out_f32 = (a.flags & PKV_FLAG_OUT_F32) != 0;
    const int tw = tid - 64;  // 0 .. 255 over the softmax warps
    constexpr int KH = kUN / 2;  // keys of a tile per thread
    constexpr int DH = D / 2;    // O columns per thread
    int xphase = 0;
    auto quarter_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(&xbar[wq]);
      return wait(&xbar[wq], (xphase++) & 1);
    };
    // half hf of this thread's row of a unit's Q (zeros past the unit's
    // tokens), the row's D / 4 columns of bf16 pairs in Q's TMEM columns
    auto q_src = [&](const XUnit &y, bool &vy) -> const uint4 * {
      const int iy = y.j * TQ + row / G;
      vy = iy < y.n;
      const long long qy = vy ? (long long)(y.q0 + iy) * Hq + y.g * G + row % G : 0;
      return reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(a.q) + qy * D +
                                             hf * (D / 2));
    };
    auto q_stage = [&](const XUnit &y) {
      bool vy;
      const uint4 *src = q_src(y, vy);
      uint32_t r[D / 4];
#pragma unroll
      for (int c = 0; c < D / 16; ++c) {
        const uint4 v = vy ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
        r[4 * c] = v.x;
        r[4 * c + 1] = v.y;
        r[4 * c + 2] = v.z;
        r[4 * c + 3] = v.w;
      }
      if constexpr (D == 128) tmem_st32(trow + kUQCol + hf * (D / 4), r);
      else tmem_st16(trow + kUQCol + hf * (D / 4), r);
    };
    // the stores landed, ordered before the tensor cores' reads: arrive on q_full
    auto q_publish = [&]() {
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_full);
    };
    bool q_pre = false;  // the current unit's Q was published with the previous unit's last P
    int k = 0;
    for (int ui = 0, u; !s_abort && (u = unit_of(ui)) >= 0; ++ui) {
      const XUnit x = xunit(a, u, TQ, jmax);
      if (!x.live) continue;
      const int T = unit_tiles(x);
      const int i = x.j * TQ + row / G;
      const bool valid = i < x.n;
      const int pos = !valid ? -1 : full_mode ? x.L - 1 : x.L - x.n + i;
      const long long qrow = valid ? (long long)(x.q0 + i) * Hq + x.g * G + row % G : 0;
      float m_used = -INFINITY, l = 0.f;
      int bad = 0;
      bool ok = true;
      if (T > 0) {
        if (!q_pre) {
          q_stage(x);
          q_publish();
        }
        // consumed here: a unit without tiles in between keeps it for the
        // next unit that has some
        q_pre = false;
      }
      bool pre = false;  // the next unit has tiles: its Q is staged behind this unit's last P
      XUnit y;
      for (int t = 0; t < T && ok; ++t) {
        const int kk = k + t, b = kk % kUSBufs;
        const int t0 = x.k0 + t * kUN + hf * KH;  // this thread's first key
        if (!wait(&s_full[b], (kk / kUSBufs) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (t == T - 1) {
          // Every Q K^T of the unit is done: the next unit's Q rows are
          // fetched into L2 now, stored into Q's columns behind this tile's
          // P and published, so the next unit's Q K^T overlaps this unit's
          // epilogue.
          for (int uj = ui + 1, u2; !pre && (u2 = unit_of(uj)) >= 0; ++uj) {
            y = xunit(a, u2, TQ, jmax);
            if (y.live && unit_tiles(y) > 0) {
              bool vy;
              const uint4 *src = q_src(y, vy);
              if (vy) asm volatile("prefetch.global.L2 [%0];" ::"l"(src));
              pre = true;
            }
          }
        }
        uint32_t sv[KH / 32][32];
#pragma unroll
        for (int c = 0; c < KH / 32; ++c) tmem_ld32(sv[c], trow + b * kUN + hf * KH + 32 * c);
        tmem_wait_ld();
        // keys past the row's position or the split's end count as -inf
        const int lim = min(pos, x.k1 - 1) - t0;
        const bool whole = lim >= KH - 1;  // every key of this half attended
        // partial row maximum in log2 units (four partial maxima, two scores
        // per 3-input max); with a positive scale the raw scores' maximum is
        // scaled once and each pair of weights is one paired FMA and two ex2
        if (!pos_scale) {
#pragma unroll
          for (int c = 0; c < KH; ++c)
            sv[c >> 5][c & 31] = __float_as_uint(__uint_as_float(sv[c >> 5][c & 31]) * qk_scale);
        }
        float mxp[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (whole) {
#pragma unroll
          for (int c = 0; c < KH; c += 2)
            mxp[(c >> 1) & 3] = fmax3(mxp[(c >> 1) & 3], __uint_as_float(sv[c >> 5][c & 31]),
                                      __uint_as_float(sv[c >> 5][(c & 31) + 1]));
        } else {
#pragma unroll
          for (int c = 0; c < KH; c += 2)
            mxp[(c >> 1) & 3] = fmax3(mxp[(c >> 1) & 3],
                                      c <= lim ? __uint_as_float(sv[c >> 5][c & 31]) : -INFINITY,
                                      c + 1 <= lim ? __uint_as_float(sv[c >> 5][(c & 31) + 1])
                                                   : -INFINITY);
        }
        float mpart = fmaxf(fmax3(mxp[0], mxp[1], mxp[2]), mxp[3]);
        if (pos_scale) mpart *= qk_scale;
        s_xmax[kk & 1][hf][row] = mpart;
        if (!quarter_sync()) {  // both halves' maxima, and both have loaded their S
          ok = false;
          break;
        }
        const float mx = fmaxf(mpart, s_xmax[kk & 1][hf ^ 1][row]);
        float alpha = 1.f;
        bool rescale = false;
        if (mx > m_used + kURescale || (m_used == -INFINITY && mx != -INFINITY)) {
          if (m_used != -INFINITY) {
            alpha = exp2f(m_used - mx);
            rescale = true;
          }
          m_used = mx;
        }
        // no key of this row attended yet: every weight is 0
        const float mref = m_used == -INFINITY ? INFINITY : m_used;
        const float fs = pos_scale ? qk_scale : 1.f;
        const uint64_t fs2 = f2(fs, fs), nm2 = f2(-mref, -mref), neg1 = f2(-1.f, -1.f);
        uint64_t sp2[4] = {0ull, 0ull, 0ull, 0ull};
        // P into the tile's S buffer, bf16 pairs (even key in the low half):
        // P_hi in its first 64 columns, P_lo (the residual e - P_hi) in the next 64
#pragma unroll
        for (int c0 = 0; c0 < KH; c0 += 32) {
          uint32_t ph[16], pl[16];
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const uint64_t x2 = f2_fma(f2(__uint_as_float(sv[c0 >> 5][c]),
                                          __uint_as_float(sv[c0 >> 5][c + 1])),
                                       fs2, nm2);
            float e0 = ex2_approx(f2_lo(x2)), e1 = ex2_approx(f2_hi(x2));
            if (!whole) {
              e0 = c0 + c <= lim ? e0 : 0.f;
              e1 = c0 + c + 1 <= lim ? e1 : 0.f;
            }
            const uint64_t e2 = f2(e0, e1);
            sp2[(c >> 1) & 3] = f2_add(sp2[(c >> 1) & 3], e2);
            const uint32_t hi = pack_bf16x2(e0, e1);
            const uint64_t r2 = f2_fma(f2(bf16lo(hi), bf16hi(hi)), neg1, e2);
            ph[c >> 1] = hi;
            pl[c >> 1] = pack_bf16x2(f2_lo(r2), f2_hi(r2));
          }
          tmem_st16(trow + b * kUN + hf * (KH / 2) + c0 / 2, ph);
          tmem_st16(trow + b * kUN + kUN / 2 + hf * (KH / 2) + c0 / 2, pl);
        }
        const uint64_t s2 = f2_add(f2_add(sp2[0], sp2[1]), f2_add(sp2[2], sp2[3]));
        const float sum = f2_lo(s2) + f2_hi(s2);
        l = l * alpha + sum;
        if (t >= 1 && __any_sync(0xffffffffu, rescale)) {
          // O holds every earlier tile once the previous tile's P V is done
          if (!wait(&buf_free[(kk - 1) % kUSBufs], ((kk - 1) / kUSBufs) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < DH; c += 32) {
            uint32_t o[32];
            tmem_ld32(o, trow + kUOCol + hf * DH + c);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(trow + kUOCol + hf * DH + c, o);
          }
        }
        if (t == T - 1) {
          // The last tile: once its V has landed, the unit's bad page bits;
          // V rows past the split's end hold what the pool or the stage's
          // previous tile held, and P = 0 does not cancel a NaN, so they are
          // cleared (its P V waits for this warp's arrival).
          const int vs = kk % kUVStages;
          if (!wait(&v_full[vs], (kk / kUVStages) & 1)) {
            ok = false;
            break;
          }
          bad |= s_ubad[ui & 3];
          const int first = x.k1 - (x.k0 + t * kUN);
          const uint32_t vb = sbase + C::OFF_V + vs * C::KBYTES;
          for (int e = tw; e < (kUN - first) * C::HALVES * 8; e += 32 * kUSoftWarps) {
            const int r = first + e / (C::HALVES * 8), rem = e % (C::HALVES * 8);
            st_shared_v4(vb + (rem >> 3) * C::KVHALF + r * 128 + (((rem & 7) ^ (r & 7)) << 4),
                         0u, 0u, 0u, 0u);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[b]);
        if (pre) {
          q_stage(y);
          q_publish();
          q_pre = true;
        }
      }
      if (!ok) break;
      // ---- the unit's rows: O / l, or the split's partial ----
      s_xsum[hf][row] = l;
      if (!quarter_sync()) break;
      const float lt = l + s_xsum[hf ^ 1][row];
      const bool zero = bad || !(lt > 0.f);
      const float inv = zero ? 0.f : 1.f / lt;
      if (T > 0) {
        const int kl = k + T - 1;  // the unit's last tile
        if (!wait(&buf_free[kl % kUSBufs], (kl / kUSBufs) & 1)) break;
        tc_fence_after();
      }
      const long long pr = qrow * a.S + x.c;
#pragma unroll
      for (int c = hf * DH; c < (hf + 1) * DH; c += 32) {
        uint32_t o[32];
        if (T > 0) {
          tmem_ld32(o, trow + kUOCol + c);
          tmem_wait_ld();
        }
        if (!valid) continue;
        float f[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) f[e] = (zero || T == 0) ? 0.f : __uint_as_float(o[e]) * inv;
        if (a.S > 1 || out_f32) {
          float *dst = a.S > 1 ? ws.o_part + pr * D + c : static_cast<float *>(a.out) + qrow * D + c;
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4 *>(dst + e) = make_float4(f[e], f[e + 1], f[e + 2], f[e + 3]);
        } else {
          uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(a.out) + qrow * D + c);
#pragma unroll
          for (int e = 0; e < 32; e += 8)
            dst[e / 8] = make_uint4(pack_bf16x2(f[e], f[e + 1]), pack_bf16x2(f[e + 2], f[e + 3]),
                                    pack_bf16x2(f[e + 4], f[e + 5]), pack_bf16x2(f[e + 6], f[e + 7]));
        }
      }
      if (valid && hf == 0) {
        if (a.S > 1) {
          // a failed split is marked l = -1: the merge writes the row as zeros
          ws.ml_part[pr * 2] = zero ? -INFINITY : m_used * kLn2;
          ws.ml_part[pr * 2 + 1] = bad ? -1.f : (zero ? 0.f : lt);
        } else if ((a.flags & PKV_FLAG_WRITE_LSE) && ws.lse) {
          ws.lse[qrow] = zero ? -INFINITY : m_used * kLn2 + logf(lt);
        }
      }
      // O's loads are done before the next unit's first P is published (its
      // first P V overwrites O); the row sums are read before they are
      // rewritten
      tc_fence_before();
      if (!quarter_sync()) break;
      k += T;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(kUTmemCols)
                 : "memory");
  }
}

template <int D, int G>
cudaError_t launch_umma_one(const XArgs &a, cudaStream_t st) {
  using C = UCfg<D>;
  static int occ_cache[64] = {0};
  static int sms_cache[64] = {0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const int di = dev & 63;
  auto kern = extend_umma_kernel<D, G>;
  if (occ_cache[di] == 0) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    int occ = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kUThreads, C::SMEM);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    sms_cache[di] = sms;
    // every resident CTA holds kUTmemCols of the SM's 512 TMEM columns
    const int tmem_cap = 512 / kUTmemCols;
    occ_cache[di] = occ < 1 ? 1 : (occ > tmem_cap ? tmem_cap : occ);
  }
  constexpr int TQ = kUM / G;
  const long long units =
      (long long)((a.max_qo_len + TQ - 1) / TQ) * a.S * a.batch * a.ws.n_kv_heads;
  if (units <= 0) return cudaSuccess;
  if (units > 0x7fffffffll) return cudaErrorInvalidValue;
  const long long cap = (long long)sms_cache[di] * occ_cache[di];
  const int grid = (int)(units < cap ? units : cap);
  CUtensorMap tmk, tmv;
  memset(&tmk, 0, sizeof(tmk));
  memset(&tmv, 0, sizeof(tmv));
  if (!xencode_pool_map(&tmk, a.ws.k_pool, a.ws, 1) || !xencode_pool_map(&tmv, a.ws.v_pool, a.ws, 1))
    return cudaErrorNotSupported;
  // Programmatic dependent launch when the grid leaves CTA slots free (its
  // start, and with PKV_FLAG_PLAN_EARLY its unit order and first cached
  // tiles, then overlap the previous kernel's end); a grid that fills every
  // slot launches plainly (measured: 46.6 against 49.4 us per launch on four
  // 256-token chunks with programmatic launch, 48.0 with the early start).
  if (grid < cap) {
    e = launch_pdl(kern, dim3(grid), dim3(kUThreads), C::SMEM, st, a, tmk, tmv);
  } else {
    XArgs b = a;  // nothing to overlap: the plain kernel
    b.flags &= ~PKV_FLAG_PLAN_EARLY;
    kern<<<grid, kUThreads, C::SMEM, st>>>(b, tmk, tmv);
    e = cudaGetLastError();
  }
  if (a.S > 1 && e == cudaSuccess) e = launch_extend_merge(a, D, st);
  return e;
}

}  // namespace

bool extend_umma_supported(const pkv_workspace &ws) {
  if (ws.n_kv_heads <= 0 || ws.n_q_heads % ws.n_kv_heads) return false;
  const int G = ws.n_q_heads / ws.n_kv_heads;
  return (ws.head_dim == 64 || ws.head_dim == 128) &&
         (G == 1 || G == 2 || G == 4 || G == 8 || G == 16) && xtma_pages(ws);
}

cudaError_t launch_extend_umma(const XArgs &a, cudaStream_t st) {
  const int D = a.ws.head_dim, G = a.ws.n_q_heads / a.ws.n_kv_heads;
#define PKV_U_CASE(DD, GG) \
  if (D == DD && G == GG) return launch_umma_one<DD, GG>(a, st);
  PKV_U_CASE(128, 1) PKV_U_CASE(128, 2) PKV_U_CASE(128, 4) PKV_U_CASE(128, 8)
  PKV_U_CASE(128, 16) PKV_U_CASE(64, 1) PKV_U_CASE(64, 2) PKV_U_CASE(64, 4)
  PKV_U_CASE(64, 8) PKV_U_CASE(64, 16)
#undef PKV_U_CASE
  return cudaErrorNotSupported;
}

}  // namespace pkv
