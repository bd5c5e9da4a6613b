// oz_gemm.cu -- steps a3 + a4: one exact integer GEMM per modulus, then mod m_t.
//
// [Ozaki II] Algorithm 1, step 3: C'_t = A'_t B'_t exactly, C''_t = C'_t mod m_t.
// The pages run this as an INT8 x INT8 -> INT32 GEMM.  sm_103a has no INT8 tcgen05
// MMA, so the same exact products run on the BF16 tensor-core path: every residue in
// [-128, 127] is exact in bf16, every product (<= 2^14) is exact, and the FP32
// accumulator in tensor memory adds integers exactly while |partial sum| <= 2^24.
// The k loop is therefore cut into chunks of 1024 (1024 * 2^14 = 2^24).  Each chunk
// starts from zero in one of two alternating TMEM accumulators; the epilogue warps read
// it (tcgen05.ld), hand the accumulator straight back to the MMA, take each value to a
// representative in (-m_t, m_t) with one FP32 quotient (exact) and add it plus m_t to
// running sums held in registers (two 16-bit lanes per register, one integer add per two
// values), which are reduced mod m_t only every 64 chunks and at the tile's end.  After the tile's last chunk the
// residues go through shared memory to coalesced 16-byte stores of the uint8 plane.
// This replaces the pages' block multiplication for k >= 2^17: the result is exact for
// every k.  The same engine in exact mode (Scheme I) converts each chunk to INT32 and
// adds it into the output, and in maximum mode (OS II-accu, one chunk holding the whole
// k) reduces the product's rows and columns to their maxima.
//
// Kernel shape: clusters of two CTAs (cta_group::2), persistent over work units
// (256 x 256 tile, modulus).  Each CTA loads its 128 rows of A and its 128 rows of B
// per 64-k stage (TMA, 128-byte swizzle, 6 stages of 32 KB) completing on the pair
// leader's mbarrier; the leader issues tcgen05.mma.cta_group::2 (M=256, N=256, K=16)
// and multicasts its commits to both CTAs; each CTA's epilogue drains its own 128
// TMEM lanes.
//   warp 0: TMA producer   warp 1: TMEM owner + MMA issuer (leader)   warps 2-9: epilogue
//   TMEM: 512 columns per CTA = two 128-lane x 256-column FP32 accumulators.
// Every mbarrier wait is bounded (oz::mbar_wait); on expiry the CTA records
// OZ_ETIMEOUT in the device status word, drains what it issued and returns.
#include <cuda.h>

#include <atomic>

#include "oz_device.cuh"
#include "oz_internal.h"

namespace oz {

namespace gemm {
// A CTA pair computes a 256 x 256 tile: each CTA holds 128 rows of A and 128 rows (the
// N dimension) of B per stage, and its 128 rows of the accumulator in its own TMEM.
constexpr int BM = 256;          // tile rows (both CTAs)
constexpr int BN = 256;          // tile columns
constexpr int HALF_M = BM / 2;   // rows per CTA
constexpr int HALF_N = BN / 2;   // B rows per CTA
constexpr int BK = 64;
constexpr int UMMA_K = 16;
constexpr int STAGES = 6;
constexpr int KB_PER_CHUNK = 16;  // 1024 k per chunk: |sum| <= 1024 * 2^14 = 2^24, exact in FP32
// Scheduling K-block: whole K.  (Shorter K-blocks make the pairs' short panels fit L2 only
// while the pairs run in lockstep; measured at 16384^3 they drift apart and DRAM reads rose
// from 248 GB to 364 GB per launch, so each unit takes the whole k range.)
constexpr int KB_PER_BLOCK = 1 << 24;
constexpr uint32_t A_STAGE = HALF_M * BK * 2;
constexpr uint32_t B_STAGE = HALF_N * BK * 2;
constexpr uint32_t STAGE_BYTES = A_STAGE + B_STAGE;
constexpr int EPI_WARPS = 8;                 // two per SM sub-partition
constexpr int EPI_THREADS = EPI_WARPS * 32;
constexpr int THREADS = 64 + EPI_THREADS;   // TMA warp, MMA warp, epilogue warps
constexpr uint32_t TMEM_COLS = 512;         // two 128-lane x 256-column FP32 accumulators
constexpr uint32_t STASH_BYTES = HALF_M * BN;  // this CTA's uint8 residue half tile, [col][row]
constexpr size_t SMEM_BYTES = 1024 /*align slack*/ + STAGES * STAGE_BYTES + STASH_BYTES + 256 /*barriers*/;
constexpr uint32_t IDESC = umma_idesc_bf16_f32(BM, BN);
static_assert(KB_PER_CHUNK * BK * 128 * 128 <= (1 << 24), "chunk too long for exact FP32 sums");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
}  // namespace gemm

__device__ int g_status = 0;

// Pair pacing (never needed for correctness).  Every kPaceEvery k-blocks a pair leader's
// producer adds 1 to its launch's counter and compares its own count with the pairs'
// average (the counter value it loaded at the previous checkpoint, so the load latency is
// hidden); a producer more than kPaceWindow checkpoints ahead pauses, for at most
// kPaceLimitNs (a pair whose pause runs out stops pausing for the rest of the launch: its
// peers are not all resident).  Pairs that share plane panels then stream them at about the
// same time, so the panels are read from DRAM once and served to the others from L2.  A finished
// pair adds a large credit so the tail of the launch never waits.  The counter slot of
// a launch is zeroed on its stream just before it starts.
constexpr int kPaceSlots = 64;
constexpr uint32_t kPaceEvery = 8;
constexpr uint32_t kPaceWindow = 1;
constexpr uint32_t kPaceDoneCredit = 1u << 24;
constexpr uint64_t kPaceLimitNs = 100000;
__device__ unsigned int g_pace_ctr[kPaceSlots];

// The epilogue's accumulator-wait limit for the launches that follow (default 4 s).
static std::atomic<unsigned long long> g_epi_wait_ns{kWaitLimitNs};
unsigned long long epilogue_wait_ns() { return g_epi_wait_ns.load(std::memory_order_relaxed); }

int* device_status_ptr() {
  int* p = nullptr;
  cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_status);
  return p;
}

// A wait expired: record it in the device status word and stop the pair (this CTA's abort
// flag and the peer's, through its shared::cluster address).
__device__ __forceinline__ void record_timeout(volatile int* abort_flag) {
  *abort_flag = 1;
  st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(abort_flag)), cluster_ctarank() ^ 1u), 1u);
  atomicExch(&g_status, OZ_ETIMEOUT);
}

// Same, for the teardown, which touches no shared memory of the peer.
__device__ __forceinline__ void record_timeout_local(volatile int* abort_flag) {
  *abort_flag = 1;
  atomicExch(&g_status, OZ_ETIMEOUT);
}

// Exact remainder of an integer-valued float v (|v| < 2^25) modulo m (173 <= m <= 256),
// in [0, m).  q is v/m rounded to an integer by the 1.5 * 2^23 magic constant (|v/m| <
// 2^22); it is floor(v/m) or one more, so v - q m is exact and lies in (-m, m).
__device__ __forceinline__ float exact_mod(float v, float m, float inv_m) {
  const float q = fmaf(v, inv_m, 12582912.0f) - 12582912.0f;
  const float r = fmaf(-q, m, v);
  return r < 0.0f ? r + m : r;
}

// v - m round(v/m) for an integer-valued float v (|v| < 2^25): exact, in (-m, m) (the
// quotient of exact_mod without its fix-up).
__device__ __forceinline__ float near_mod(float v, float m, float inv_m) {
  const float q = fmaf(v, inv_m, 12582912.0f) - 12582912.0f;
  return fmaf(-q, m, v);
}

// Chunks a 16-bit running lane can take between reductions: each adds less than 2m <= 512
// to a lane that starts below m <= 256, and 256 + 64 * 511 < 2^16.
constexpr int kLaneChunks = 64;

// Reduces both 16-bit lanes of every register mod m (a lane < 2^16 is exact in FP32).
__device__ __forceinline__ void reduce_lanes(uint32_t (&run)[64], float m, float inv_m) {
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    const float lo = exact_mod(static_cast<float>(run[i] & 0xFFFFu), m, inv_m);
    const float hi = exact_mod(static_cast<float>(run[i] >> 16), m, inv_m);
    run[i] = __byte_perm(__float_as_uint(lo + 8388608.0f), __float_as_uint(hi + 8388608.0f), 0x5410);
  }
}

// Rendezvous of the epilogue warps on an mbarrier (one arrival per warp), with the same
// bounded wait as every other wait in the kernel.  Returns false on expiry.
// The warp's lanes agree on the outcome (a lane that saw the phase complete while another
// gave up follows the one that gave up), so warp-wide instructions stay converged.
__device__ __forceinline__ bool epilogue_sync(uint64_t* bar, uint32_t& phase, const volatile int* abort) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
  const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait_or_abort(bar, phase, kWaitLimitNs, abort));
  phase ^= 1;
  return ok;
}

// The epilogue's wait for an accumulator, with the launch's limit, agreed by the warp.
__device__ __forceinline__ bool epilogue_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns,
                                              const volatile int* abort) {
  return __all_sync(0xFFFFFFFFu, mbar_wait_or_abort(bar, parity, limit_ns, abort));
}

struct UnitCoord {
  int t, tm, tn;
};

__device__ __forceinline__ UnitCoord unit_coord(int u, int tiles_m, int tiles_n) {
  // modulus outermost (all CTAs share a modulus' planes), then groups of 8 row tiles
  // swept along the column tiles for L2 reuse of B.
  const int per_t = tiles_m * tiles_n;
  UnitCoord c;
  c.t = u / per_t;
  int r = u - c.t * per_t;
  const int group = 8;
  const int gsize = group * tiles_n;
  const int g = r / gsize;
  const int first_m = g * group;
  const int gm = min(group, tiles_m - first_m);
  const int in = r - g * gsize;
  c.tm = first_m + in % gm;
  c.tn = in / gm;
  return c;
}

// Work order of one CTA pair.  Its (tile, product) units are r = pair, pair + npairs, ...;
// they are taken in groups of kGroup, and within a group K-block by K-block (every unit of
// the group for K-block 0, then K-block 1, ...).  A K-block is kbb k-blocks of 64, so the
// planes a wave of pairs touches at once are short panels that stay in L2, and the K-blocks
// of one tile always follow each other on the same pair (their partial results are
// combined in program order).
constexpr int kGroup = 8;

struct PairSchedule {
  int pair, npairs, n_r, KB;
  __device__ PairSchedule(int units, int nkb, int kbb) {
    pair = static_cast<int>(blockIdx.x >> 1);
    npairs = static_cast<int>(gridDim.x >> 1);
    n_r = (units - pair + npairs - 1) / npairs;
    KB = (nkb + kbb - 1) / kbb;
  }
  __device__ int count() const { return n_r * KB; }
  __device__ void at(int idx, int& r, int& kb) const {
    const int full = n_r / kGroup * kGroup;  // units in complete groups
    int j;
    if (idx < full * KB) {
      const int g = idx / (kGroup * KB);
      const int rem = idx - g * kGroup * KB;
      kb = rem / kGroup;
      j = g * kGroup + rem % kGroup;
    } else {
      const int gsz = n_r - full;
      const int rem = idx - full * KB;
      kb = rem / gsz;
      j = full + rem % gsz;
    }
    r = pair + j * npairs;
  }
};

constexpr int kModeResidue = 0;  // Scheme II: C''_t = (A'_t B'_t) mod m_t, uint8 output
constexpr int kModeExact = 1;    // Scheme I: exact INT32 slice products
constexpr int kModeMax = 2;      // OS II-accu: row and column maxima of one exact product
constexpr int kModeExactAcc = 3; // Scheme I products of several exact chunks: INT32 sums in shared memory

// Shared-memory layout per mode.  The running-sum mode keeps half of each thread's INT32
// running sums in registers and half in a 64 KB shared-memory tile (this CTA's 128 rows x
// 128 of its 256 columns), which costs one of the six stages; each product's chunks are
// summed on chip and the output is written once.
template <int MODE>
struct ModeLayout {
  static constexpr int STAGES = (MODE == kModeExactAcc) ? 5 : gemm::STAGES;
  static constexpr uint32_t STASH = (MODE == kModeExactAcc) ? gemm::HALF_M * (gemm::BN / 2) * 4 : gemm::STASH_BYTES;
  static constexpr size_t SMEM = 1024 /*align slack*/ + STAGES * gemm::STAGE_BYTES + STASH + 256 /*barriers*/;
  static_assert(SMEM <= 232448, "shared memory budget");
};

template <int MODE>
__global__ void __launch_bounds__(gemm::THREADS, 1)
    residue_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const GemmConsts c, void* __restrict__ out_ptr, int mp, int np, int nkb) {
  using namespace gemm;
  constexpr int kStages = ModeLayout<MODE>::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * A_STAGE;
  uint8_t* stash = smem + kStages * STAGE_BYTES;  // [128 cols][128 rows]... see epilogue
  uint64_t* bars = reinterpret_cast<uint64_t*>(stash + ModeLayout<MODE>::STASH);
  uint64_t* full = bars;                  // [kStages]  TMA (both CTAs) -> MMA   (used in the leader)
  uint64_t* empty = bars + kStages;        // [kStages]  MMA -> TMA               (both CTAs)
  uint64_t* accfull = bars + 2 * kStages;  // [2]       MMA -> epilogue          (both CTAs)
  uint64_t* accempty = accfull + 2;       // [2]       epilogues (both) -> MMA  (used in the leader)
  uint64_t* drain = accempty + 2;         // [1]       all MMAs of the pair done (both CTAs)
  uint64_t* epibar = drain + 1;           // [1]       epilogue warps rendezvous (per CTA)
  uint64_t* exitbar = epibar + 1;         // [1]       the peer has finished (per CTA)
  uint64_t* proddone = exitbar + 1;       // [1]       both producers have stopped (used in the leader)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(proddone + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile uint32_t* issued_by = reinterpret_cast<volatile uint32_t*>(abort_flag + 1);  // [2] (leader)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();      // 0 = leader of the pair, 1 = peer
  const int tiles_m = mp / BM, tiles_n = np / BN;
  const int units = tiles_m * tiles_n * c.s;
  const int kbc = c.kb_per_chunk;
  const int kbb = c.kb_per_block;
  const PairSchedule sched(units, nkb, kbb);

  if (threadIdx.x == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&full[i], 2);  // one arrival (with its bytes) from each CTA's producer
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&accfull[i], 1);
      mbar_init(&accempty[i], 2 * EPI_WARPS);  // every epilogue warp of both CTAs
    }
    mbar_init(drain, 1);
    mbar_init(epibar, EPI_WARPS);
    mbar_init(exitbar, 1);
    mbar_init(proddone, 2);  // one arrival from each CTA's producer, after its last copy
    *abort_flag = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barrier initialisation visible to the peer before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ TMA producer (both CTAs)
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      const bool pacer = (rank == 0);  // the leader's producer counts the pair's progress
      bool may_pause = pacer;          // cleared once a pause runs out (see below)
      unsigned int* ctr = &g_pace_ctr[c.launch_id % kPaceSlots];
      uint32_t paced = 0, checkpoints = 0, seen = 0;
      for (int idx = 0; idx < sched.count() && !*abort_flag; ++idx) {
        int u, kblk;
        sched.at(idx, u, kblk);
        const UnitCoord uc = unit_coord(u, tiles_m, tiles_n);
        const int pa = (MODE == kModeResidue) ? uc.t : c.a_plane[uc.t];
        const int pb = (MODE == kModeResidue) ? uc.t : c.b_plane[uc.t];
        const int rowA = uc.tm * BM + static_cast<int>(rank) * HALF_M;
        const int rowB = uc.tn * BN + static_cast<int>(rank) * HALF_N;
        const int kb_end = min(nkb, (kblk + 1) * kbb);
        for (int kb = kblk * kbb; kb < kb_end; ++kb) {
          if (*abort_flag) break;  // the pair has stopped: issue nothing more
          if (!mbar_wait_or_abort(&empty[stage], phase ^ 1, kWaitLimitNs, abort_flag)) {
            if (!*abort_flag) record_timeout(abort_flag);
            break;
          }
          const uint32_t full_leader = mapa_shared(smem_u32(&full[stage]), 0);
          mbar_arrive_expect_tx_cluster(full_leader, STAGE_BYTES);
          tma_load_3d_pair(sA + stage * A_STAGE, &tmA, full_leader, kb * BK, rowA, pa);
          tma_load_3d_pair(sB + stage * B_STAGE, &tmB, full_leader, kb * BK, rowB, pb);
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
          if (pacer && ++paced % kPaceEvery == 0) {
            ++checkpoints;
            atomicAdd(ctr, 1u);
            const uint32_t np = static_cast<uint32_t>(sched.npairs);
            if (may_pause && checkpoints * np > seen + kPaceWindow * np) {  // ahead of the average: pause
              const uint64_t t0 = globaltimer_ns();
              while (checkpoints * np > seen + kPaceWindow * np && globaltimer_ns() - t0 < kPaceLimitNs) {
                __nanosleep(256);
                seen = *reinterpret_cast<volatile unsigned int*>(ctr);
              }
              // Still ahead after the limit: some pairs of this launch are not running (another
              // kernel holds their SMs), so the average cannot catch up.  Stop pausing for the
              // rest of the launch; the pair keeps counting so the others' average stays right.
              if (checkpoints * np > seen + kPaceWindow * np) may_pause = false;
            }
            seen = *reinterpret_cast<volatile unsigned int*>(ctr);  // used at the next checkpoint
          }
        }
      }
      if (pacer) atomicAdd(ctr, kPaceDoneCredit);  // finished: nobody waits for this pair
      // Every issued copy must have landed before the pair may exit.  The copies complete on
      // the leader's barriers: tell the leader's MMA thread how many stages this CTA filled
      // (it waits for any it did not consume, below), then, on the normal path, wait for
      // this CTA's last stages to be released by the MMAs that read them.
      st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<uint32_t*>(&issued_by[rank])), 0),
                            static_cast<uint32_t>(issued));
      mbar_arrive_release_cluster(mapa_shared(smem_u32(proddone), 0));
      if (!*abort_flag) {
        for (int i = 0; i < kStages && i < issued; ++i) {
          if (--stage < 0) {
            stage = kStages - 1;
            phase ^= 1;
          }
          if (!mbar_wait_or_abort(&empty[stage], phase, kWaitLimitNs, abort_flag)) {
            if (!*abort_flag) record_timeout(abort_flag);
            break;
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------------------------------------ MMA issuer (leader only)
      int stage = 0;
      uint32_t phase = 0;
      uint32_t g = 0;  // chunk counter: accumulator g & 1
      uint32_t consumed = 0;  // stages whose copies this thread has waited for
      bool ok = true;
      for (int idx = 0; idx < sched.count() && ok && !*abort_flag; ++idx) {
        int u, kblk;
        sched.at(idx, u, kblk);
        const int kb_begin = kblk * kbb, kb_end = min(nkb, kb_begin + kbb);
        const int nchunks = (kb_end - kb_begin + kbc - 1) / kbc;
        for (int ch = 0; ch < nchunks && ok; ++ch, ++g) {
          const uint32_t acc = g & 1;
          if (!mbar_wait_or_abort(&accempty[acc], ((g >> 1) & 1) ^ 1, kWaitLimitNs, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + acc * BN;
          const int kb0 = kb_begin + ch * kbc;
          const int kb1 = min(kb_end, kb0 + kbc);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!mbar_wait_or_abort(&full[stage], phase, kWaitLimitNs, abort_flag)) {
              ok = false;
              break;
            }
            ++consumed;
            tc_fence_after();
            const uint32_t a_addr = smem_u32(sA + stage * A_STAGE);
            const uint32_t b_addr = smem_u32(sB + stage * B_STAGE);
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk) {
              const uint64_t ad = umma_desc_k128(a_addr + kk * UMMA_K * 2);
              const uint64_t bd = umma_desc_k128(b_addr + kk * UMMA_K * 2);
              // every chunk starts afresh; the epilogue combines the chunks (mod m_t in
              // residue mode, exactly in INT32 in exact mode)
              const uint32_t accumulate = (kb > kb0 || kk > 0) ? 1u : 0u;
              umma_bf16_pair(d_tmem, ad, bd, IDESC, accumulate);
            }
            umma_commit_pair(&empty[stage], 0x3);  // frees the stage in both CTAs
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1;
            }
          }
          if (!ok) break;
          umma_commit_pair(&accfull[acc], 0x3);  // the chunk is in both CTAs' TMEM
        }
      }
      if (!ok && !*abort_flag) record_timeout(abort_flag);
      // Account for every copy before the pair may exit: once both producers have stopped
      // (and published how many stages they filled), wait for each stage filled after the
      // last one consumed here, arriving for a producer that stopped before filling it, so
      // that its phase completes exactly when the copies that were issued have landed.
      // (On the normal path both producers filled exactly the stages consumed here.)
      if (mbar_wait_acquire_cluster(proddone, 0)) {
        const uint32_t n0 = issued_by[0], n1 = issued_by[1];
        const uint32_t top = n0 > n1 ? n0 : n1;
        for (uint32_t q = consumed; q < top && q < consumed + kStages; ++q) {  // at most kStages are in flight
          const int st = static_cast<int>(q % kStages);
          if (q >= n0) mbar_arrive(&full[st]);
          if (q >= n1) mbar_arrive(&full[st]);
          if (!mbar_wait(&full[st], (q / kStages) & 1)) {
            record_timeout(abort_flag);
            break;
          }
        }
      } else {
        record_timeout(abort_flag);
      }
      umma_commit_pair(drain, 0x3);  // arrives in both CTAs once every MMA above is done
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2-9, both CTAs)
    // Thread = one accumulator row (TMEM lane) of this CTA's 128 rows and one half of the
    // 256 columns.
    const int quad = warp & 3;             // TMEM lanes 32*quad .. 32*quad+31
    const int half = (warp - 2) >> 2;      // columns [128*half, 128*half + 128)
    const int row = quad * 32 + lane;
    const int etid = threadIdx.x - 64;     // 0 .. EPI_THREADS-1
    const long long plane = static_cast<long long>(np) * mp;
    const int row_off = static_cast<int>(rank) * HALF_M;  // this CTA's rows of the tile
    uint32_t g = 0, eph = 0;
    bool ok = true;
    if (MODE == kModeMax) {
      // One chunk per unit (the launcher makes the whole k one chunk), so the accumulator
      // holds the tile's exact non-negative integer sums; their FP32 bit patterns order
      // like the values, so maxima are taken on the bits.
      uint32_t* rho = static_cast<uint32_t*>(out_ptr);  // [mp] row maxima, then [np] column maxima
      uint32_t* gamma = rho + mp;
      for (int idx = 0; idx < sched.count() && ok; ++idx, ++g) {
        int u, kblk;
        sched.at(idx, u, kblk);
        const UnitCoord uc = unit_coord(u, tiles_m, tiles_n);
        const uint32_t acc = g & 1;
        if (!epilogue_wait(&accfull[acc], (g >> 1) & 1, c.epi_wait_ns, abort_flag)) {
          ok = false;
          if (lane == 0 && !*abort_flag) record_timeout(abort_flag);
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN + half * 128;
        const int col0 = uc.tn * BN + half * 128;
        uint32_t rmax = 0;
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
          uint32_t v[32];
          tmem_ld32(taddr + cb * 32, v);
          tmem_ld_wait();
          if (cb == 3) {  // the whole tile is in registers: hand the accumulator back
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&accempty[acc]), 0));
          }
          uint32_t mine = 0;  // maximum of column col0 + cb * 32 + lane over this warp's 32 rows
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            rmax = max(rmax, v[i]);
            const uint32_t cm = __reduce_max_sync(0xFFFFFFFFu, v[i]);
            if (lane == i) mine = cm;
          }
          atomicMax(gamma + col0 + cb * 32 + lane, mine);
        }
        atomicMax(rho + uc.tm * BM + row_off + row, rmax);
      }
    } else if (MODE == kModeExactAcc) {
      // This thread's 128 columns (its row, columns half*128 .. +127): the first 64 running
      // sums live in registers, the other 64 in the shared tile, laid out [column][row] so a
      // warp's 32 rows are 32 consecutive words.  Owned by this thread alone: no barrier.
      // Units cover the whole k range (one K-block).
      int32_t* outp = static_cast<int32_t*>(out_ptr);
      int32_t* mine = reinterpret_cast<int32_t*>(stash) + (half * 64) * HALF_M + row;
      for (int idx = 0; idx < sched.count() && ok; ++idx) {
        int u, kblk;
        sched.at(idx, u, kblk);
        const int kb_begin = kblk * kbb, kb_end = min(nkb, kb_begin + kbb);
        const int nchunks = (kb_end - kb_begin + kbc - 1) / kbc;
        const UnitCoord uc = unit_coord(u, tiles_m, tiles_n);
        int32_t run[64];
        for (int ch = 0; ch < nchunks; ++ch, ++g) {
          const uint32_t acc = g & 1;
          if (!epilogue_wait(&accfull[acc], (g >> 1) & 1, c.epi_wait_ns, abort_flag)) {
            ok = false;
            if (lane == 0 && !*abort_flag) record_timeout(abort_flag);
            break;
          }
          tc_fence_after();
          const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN + half * 128;
          uint32_t v[2][32];
          tmem_ld32(taddr, v[0]);
          tmem_ld32(taddr + 32, v[1]);
          tmem_ld_wait();
#pragma unroll
          for (int c2 = 0; c2 < 64; ++c2) {
            const int32_t x = __float2int_rn(__uint_as_float(v[c2 >> 5][c2 & 31]));  // exact integer
            run[c2] = (ch == 0) ? x : run[c2] + x;
          }
          tmem_ld32(taddr + 64, v[0]);
          tmem_ld32(taddr + 96, v[1]);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&accempty[acc]), 0));
#pragma unroll
          for (int c2 = 0; c2 < 64; ++c2) {
            const int32_t x = __float2int_rn(__uint_as_float(v[c2 >> 5][c2 & 31]));
            int32_t* p = mine + c2 * HALF_M;
            *p = (ch == 0) ? x : *p + x;
          }
        }
        if (!ok) break;
        int32_t* base =
            outp + uc.t * plane + static_cast<long long>(uc.tn * BN + half * 128) * mp + uc.tm * BM + row_off + row;
#pragma unroll
        for (int c2 = 0; c2 < 64; ++c2) base[static_cast<long long>(c2) * mp] = run[c2];
#pragma unroll 8
        for (int c2 = 0; c2 < 64; ++c2) base[static_cast<long long>(64 + c2) * mp] = mine[c2 * HALF_M];
      }
    } else if (MODE == kModeExact) {
      int32_t* outp = static_cast<int32_t*>(out_ptr);
      for (int idx = 0; idx < sched.count() && ok; ++idx) {
        int u, kblk;
        sched.at(idx, u, kblk);
        const int kb_begin = kblk * kbb, kb_end = min(nkb, kb_begin + kbb);
        const int nchunks = (kb_end - kb_begin + kbc - 1) / kbc;
        const UnitCoord uc = unit_coord(u, tiles_m, tiles_n);
        int32_t* base =
            outp + uc.t * plane + static_cast<long long>(uc.tn * BN + half * 128) * mp + uc.tm * BM + row_off + row;
        for (int ch = 0; ch < nchunks; ++ch, ++g) {
          const uint32_t acc = g & 1;
          if (!epilogue_wait(&accfull[acc], (g >> 1) & 1, c.epi_wait_ns, abort_flag)) {
            ok = false;
            if (lane == 0 && !*abort_flag) record_timeout(abort_flag);
            break;
          }
          tc_fence_after();
          const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN + half * 128;
          // the whole chunk into registers first, so the accumulator goes back to the MMA
          // before the (slower) INT32 updates of the output
          uint32_t v[4][32];
#pragma unroll
          for (int cb = 0; cb < 4; ++cb) tmem_ld32(taddr + cb * 32, v[cb]);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&accempty[acc]), 0));
          const bool first = (kblk == 0 && ch == 0);
#pragma unroll
          for (int cb = 0; cb < 4; ++cb) {
            int32_t* o = base + static_cast<long long>(cb * 32) * mp;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              int32_t x = __float2int_rn(__uint_as_float(v[cb][i]));  // exact integer
              if (!first) x += o[static_cast<long long>(i) * mp];
              o[static_cast<long long>(i) * mp] = x;
            }
          }
        }
      }
    } else {
      uint8_t* C_res = static_cast<uint8_t*>(out_ptr);
      for (int idx = 0; idx < sched.count() && ok; ++idx) {
        int u, kblk;
        sched.at(idx, u, kblk);
        const int kb_begin = kblk * kbb, kb_end = min(nkb, kb_begin + kbb);
        const int nchunks = (kb_end - kb_begin + kbc - 1) / kbc;
        const UnitCoord uc = unit_coord(u, tiles_m, tiles_n);
        const float mf = c.modf[uc.t], inv = c.invf[uc.t];
        const float bias = mf + 8388608.0f;  // r + m + 2^23: its low bits are the integer r + m
        // Running sums of this thread's 128 columns, two per register (16-bit lanes).  Each
        // chunk adds r + m with r = v - m round(v/m) in (-m, m), i.e. less than 2m <= 512 per
        // lane; reducing the lanes mod m every kLaneChunks chunks keeps them below 2^16.
        uint32_t run[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) run[i] = 0;
        for (int ch = 0; ch < nchunks; ++ch, ++g) {
          const uint32_t acc = g & 1;
          if (!epilogue_wait(&accfull[acc], (g >> 1) & 1, c.epi_wait_ns, abort_flag)) {
            ok = false;
            if (lane == 0 && !*abort_flag) record_timeout(abort_flag);
            break;
          }
          tc_fence_after();
          const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + acc * BN + half * 128;
#pragma unroll
          for (int cb = 0; cb < 4; ++cb) {
            uint32_t v[32];
            tmem_ld32(taddr + cb * 32, v);
            tmem_ld_wait();
            if (cb == 3) {  // the whole chunk is in registers: hand the accumulator back
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&accempty[acc]), 0));
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float r0 = near_mod(__uint_as_float(v[2 * i]), mf, inv) + bias;
              const float r1 = near_mod(__uint_as_float(v[2 * i + 1]), mf, inv) + bias;
              run[cb * 16 + i] += __byte_perm(__float_as_uint(r0), __float_as_uint(r1), 0x5410);
            }
          }
          // keep the lanes below 2^16; after the last chunk every lane is in [0, m)
          if ((ch + 1) % kLaneChunks == 0 || ch + 1 == nchunks) reduce_lanes(run, mf, inv);
        }
        if (!ok) break;
        // This K-block's residues join the tile's running result in the stash ([col][row]
        // bytes): for later K-blocks the previous result is first read back from the plane
        // (16-byte loads, each thread the chunks it stored), then coalesced 16-byte stores.
        uint8_t* dst = C_res + uc.t * plane + static_cast<long long>(uc.tn) * BN * mp + uc.tm * BM + row_off;
        const uint32_t mi = static_cast<uint32_t>(mf);
        if (kblk > 0) {
#pragma unroll
          for (int i = 0; i < (BN * HALF_M / 16) / EPI_THREADS; ++i) {
            const int q = etid + i * EPI_THREADS;
            const int col = q >> 3, part = q & 7;
            *reinterpret_cast<uint4*>(stash + col * HALF_M + part * 16) =
                *reinterpret_cast<const uint4*>(dst + static_cast<long long>(col) * mp + part * 16);
          }
          if (!epilogue_sync(epibar, eph, abort_flag)) {
            if (lane == 0 && !*abort_flag) record_timeout(abort_flag);
            break;
          }
        }
        uint8_t* col0 = stash + (half * 128) * HALF_M + row;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          uint32_t lo = run[i] & 0xFFFFu, hi = run[i] >> 16;
          if (kblk > 0) {
            lo += col0[(2 * i) * HALF_M];
            hi += col0[(2 * i + 1) * HALF_M];
            lo = (lo >= mi) ? lo - mi : lo;
            hi = (hi >= mi) ? hi - mi : hi;
          }
          col0[(2 * i) * HALF_M] = static_cast<uint8_t>(lo);
          col0[(2 * i + 1) * HALF_M] = static_cast<uint8_t>(hi);
        }
        if (!epilogue_sync(epibar, eph, abort_flag)) {
          if (lane == 0 && !*abort_flag) record_timeout(abort_flag);
          break;
        }

#pragma unroll
        for (int i = 0; i < (BN * HALF_M / 16) / EPI_THREADS; ++i) {
          const int q = etid + i * EPI_THREADS;
          const int col = q >> 3, part = q & 7;
          *reinterpret_cast<uint4*>(dst + static_cast<long long>(col) * mp + part * 16) =
              *reinterpret_cast<const uint4*>(stash + col * HALF_M + part * 16);
        }
        if (!epilogue_sync(epibar, eph, abort_flag)) {
          if (lane == 0 && !*abort_flag) record_timeout(abort_flag);
          break;
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) {
    // every MMA of the pair (and every commit before it) has completed ...
    if (!mbar_wait(drain, 0)) record_timeout_local(abort_flag);
    // ... and the peer is done with this CTA's barriers and shared memory
    mbar_arrive_cluster(mapa_shared(smem_u32(exitbar), rank ^ 1u));
    if (!mbar_wait(exitbar, 0)) record_timeout_local(abort_flag);
  }
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

// ------------------------------------------------------------------ host side
typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                     const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                     CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static PFN_encodeTiled get_encode_fn() {
  static PFN_encodeTiled fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_encodeTiled>(p);
  }
  return fn;
}

// 3-D map over planes [s][rows][kp] of bf16, box {64, box_rows, 1}, 128-byte swizzle.
static bool make_plane_map(CUtensorMap* map, const void* base, int s, int rows, int kp, int box_rows) {
  PFN_encodeTiled enc = get_encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kp), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(s)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kp) * 2, static_cast<cuuint64_t>(kp) * 2 * rows};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(gemm::BK), static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Exact chunks per product from which the slice GEMM keeps its running sums on chip (five
// stages instead of six) rather than folding every chunk into the output through L2.
constexpr int kAccChunks = 2;

static uint32_t next_launch_id() {
  static uint32_t id = 0;
  return __atomic_add_fetch(&id, 1u, __ATOMIC_RELAXED);
}

template <int MODE>
static int launch_gemm(int mp, int np, int kp, int a_planes, int b_planes, const GemmConsts& c,
                       const uint16_t* A_planes, const uint16_t* B_planes, void* out, cudaStream_t stream) {
  using namespace gemm;
  if (mp % BM || np % BN || kp % BK || c.kb_per_chunk < 1 || c.kb_per_block < c.kb_per_chunk ||
      c.kb_per_block % c.kb_per_chunk)
    return OZ_EINVAL;
  CUtensorMap tmA, tmB;
  if (!make_plane_map(&tmA, A_planes, a_planes, mp, kp, HALF_M)) return OZ_ECUDA;
  if (!make_plane_map(&tmB, B_planes, b_planes, np, kp, HALF_N)) return OZ_ECUDA;
  if (cudaFuncSetAttribute(residue_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(ModeLayout<MODE>::SMEM)) != cudaSuccess)
    return OZ_ECUDA;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return OZ_ECUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return OZ_ECUDA;
  const long long units = static_cast<long long>(mp / BM) * (np / BN) * c.s;
  const int pairs = static_cast<int>(units < sms / 2 ? units : sms / 2);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  cfg.blockDim = dim3(THREADS, 1, 1);
  cfg.dynamicSmemBytes = ModeLayout<MODE>::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const int nkb = kp / BK;
  GemmConsts cl = c;
  cl.launch_id = next_launch_id();
  cl.epi_wait_ns = epilogue_wait_ns();
  {  // zero this launch's pacing counter on the stream
    unsigned int* ctr = nullptr;
    if (cudaGetSymbolAddress(reinterpret_cast<void**>(&ctr), g_pace_ctr) != cudaSuccess) return OZ_ECUDA;
    if (cudaMemsetAsync(ctr + cl.launch_id % kPaceSlots, 0, sizeof(unsigned int), stream) != cudaSuccess)
      return OZ_ECUDA;
  }
  if (cudaLaunchKernelEx(&cfg, residue_gemm_kernel<MODE>, tmA, tmB, cl, out, mp, np, nkb) != cudaSuccess)
    return OZ_ECUDA;
  return cudaGetLastError() == cudaSuccess ? OZ_OK : OZ_ECUDA;
}

int launch_residue_gemm(int mp, int np, int kp, const GemmConsts& c, const uint16_t* A_planes,
                        const uint16_t* B_planes, uint8_t* C_res, cudaStream_t stream) {
  GemmConsts cc = c;
  cc.kb_per_chunk = gemm::KB_PER_CHUNK;
  cc.kb_per_block = gemm::KB_PER_BLOCK;
  return launch_gemm<kModeResidue>(mp, np, kp, c.s, c.s, cc, A_planes, B_planes, C_res, stream);
}

int launch_slice_gemm(int mp, int np, int kp, int a_planes, int b_planes, const GemmConsts& c,
                      const uint16_t* A_planes, const uint16_t* B_planes, int32_t* out, cudaStream_t stream) {
  const int nkb = kp / gemm::BK;
  const int chunks = c.kb_per_chunk > 0 ? (nkb + c.kb_per_chunk - 1) / c.kb_per_chunk : 1;
  if (chunks >= kAccChunks && c.kb_per_block >= nkb)
    return launch_gemm<kModeExactAcc>(mp, np, kp, a_planes, b_planes, c, A_planes, B_planes, out, stream);
  return launch_gemm<kModeExact>(mp, np, kp, a_planes, b_planes, c, A_planes, B_planes, out, stream);
}

int launch_bound_gemm(int mp, int np, int kp, const uint16_t* A_plane, const uint16_t* B_plane, uint32_t* maxes,
                      cudaStream_t stream) {
  GemmConsts c{};
  c.s = 1;
  c.kb_per_chunk = kp / gemm::BK;  // the whole k in one chunk: the caller keeps q 4^b <= 2^24
  c.kb_per_block = c.kb_per_chunk;
  c.a_plane[0] = 0;
  c.b_plane[0] = 0;
  if (cudaMemsetAsync(maxes, 0, sizeof(uint32_t) * (static_cast<size_t>(mp) + np), stream) != cudaSuccess)
    return OZ_ECUDA;
  return launch_gemm<kModeMax>(mp, np, kp, 1, 1, c, A_plane, B_plane, maxes, stream);
}

}  // namespace oz

extern "C" int ozaki_set_epilogue_wait_ns(long long ns) {
  if (ns < -1) return OZ_EINVAL;
  oz::g_epi_wait_ns.store(ns == -1 ? oz::kWaitLimitNs : static_cast<unsigned long long>(ns),
                          std::memory_order_relaxed);
  return OZ_OK;
}
