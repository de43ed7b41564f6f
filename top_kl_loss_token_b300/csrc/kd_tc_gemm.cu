// kd_tc_gemm.cu -- the tensor-core kernels of the fused top-K KL loss and of
// the other paths built on it.
//
// One persistent, warp-specialised kernel template runs every contraction on
// the tcgen05 tensor cores ("Efficient Knowledge Distillation for LLMs:
// Offline Top-K Logits and a Fused Chunked KL Loss", ai2day.live story, "What
// did the researchers change?": the logits are produced and consumed one chunk
// of the sequence at a time, never as the full grid).  The launch modes:
//
//   pass 1     z = h_c W^T for one token chunk (M = chunk rows, N = V, K = d);
//              the epilogue turns each 128 x 128 quarter of the fp32
//              accumulator into logsumexp statistics (block max, sum of
//              exponentials, teacher-weighted logit sum) and, when the
//              gradients follow, stores the normalised exponentials
//              u = 2^(s2 - m2) as bf16;
//   backward   grad_h rows of the chunk = G_c W   (M = chunk, N = d, K = V) and
//              grad_W (+)= G_c^T h_c              (M = V, N = d, K = chunk),
//              both in the same launch, fp32 results stored or accumulated
//              (also the plain GEMM of kd_umma_gemm_bf16);
//   top-K      the teacher top-K cache: the largest rank key of every
//              128-column block of a leading sample of the vocabulary (first
//              pass), then over all of it every block's largest key and the
//              keys reaching each row's threshold (second pass; run again,
//              gated, for rows whose candidates overflowed);
//   dual       the full-vocabulary loss: the teacher's and the student's
//              logits of the same tile into the two accumulators, their block
//              statistics and both sets of stored exponentials.
//
// The kernel runs as clusters of two CTAs ("CTA pairs", one CTA per SM).  A
// pair owns a 256-row output tile: each CTA stages its 128 rows of A and half
// of the tile's B columns, and one tcgen05.mma.cta_group::2 issued by the
// pair's first CTA multiplies the whole 256 x N tile, each CTA's tensor
// memory receiving its own 128 rows.  Staging half of B per SM halves the
// operand bytes per stage, so 7 stages of 64-deep K blocks fit in shared
// memory.
//
// CTA layout (352 threads):
//   warp 0      TMA producer of A.  In the first CTA it also takes tile
//               numbers from a global counter and hands them to every role of
//               both CTAs through a shared-memory ring;
//   warp 10     TMA producer of B.  Both CTAs' producers stream their halves
//               of each K block into a 7-stage ring whose "full" barrier lives
//               in the first CTA.  A and B are issued from separate warps
//               because one thread issuing every tensor copy of a stage in
//               turn cannot keep the pair's MMA fed;
//   warp 1      allocates TMEM for the pair (two 128 x 256 fp32 accumulators
//               per CTA); in the first CTA one lane issues the pair MMAs
//               (256 x N x 16, bf16 in, fp32 out);
//   warps 2-9   epilogue: each warp reads 32 TMEM lanes (rows) x 128 columns
//               of its own CTA's accumulator.  Large contiguous outputs (pass
//               1's stored exponentials, plain GEMM results) go out through a
//               4 KiB staging buffer per warp and TMA stores (adds when
//               accumulating), 32 rows x 128 bytes per store; those modes keep
//               6 ring stages instead of 7 to make room.
// Operands are staged in the 128-byte swizzle layout; a K-major operand tile
// is one TMA box of 64 x rows, an MN-major tile is made of 64 x 64 atoms,
// brought by one 3-D box when the tile starts on an atom boundary.
// Every wait is time-bounded (kd_ptx.cuh): on a timeout the CTA records
// KD_FLAG_TIMEOUT, tells the other CTA of the pair, drains its in-flight
// copies and MMAs, frees TMEM and exits.
#include <math.h>
#include <string.h>

#include "kd_internal.h"
#include "kd_ptx.cuh"

namespace kd {
namespace {

constexpr int kEpiWarps = 8;
constexpr int kBProducerWarp = 2 + kEpiWarps;    // warp 10
constexpr int kThreads = (3 + kEpiWarps) * 32;
constexpr int kSched = 4;
constexpr int kMaxStages = 7;
constexpr int kPairM = 2 * kBM;                 // rows of a pair's output tile
constexpr uint32_t kTmemCols = 2 * kBN;
constexpr int kABytes = kBM * kBK * 2;          // this CTA's 128 rows of A
constexpr int kBBytes = (kBN / 2) * kBK * 2;    // this CTA's half of B (at most)
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kAtomBytes = 64 * kBK * 2;  // one 64 (MN) x 64 (K) box of an MN-major tile

// Barriers and the tile ring.  In the pair's second CTA, full[], tempty[] and
// sempty[] are unused: those waits happen in the first CTA.
struct Ctl {
  uint64_t full[kMaxStages];   // first CTA: both CTAs' operands of a stage landed
  uint64_t empty[kMaxStages];  // each CTA: the pair MMAs reading a stage are done
  uint64_t tfull[2];        // each CTA: accumulator b is complete
  uint64_t tempty[2];       // first CTA: both CTAs' epilogues have read accumulator b
  uint64_t sfull[kSched];   // each CTA: a tile number is in sched_tile[slot]
  uint64_t sempty[kSched];  // first CTA: every role of both CTAs has taken it
  uint64_t drain;
  int sched_tile[kSched];
  uint32_t tmem_base;
  int abort;
};

enum : int {
  kModePass1 = 0,     // student logits + top-K statistics (the loss against the cache)
  kModeStore = 1,     // plain GEMMs, fp32 results stored or accumulated
  kModeTopkMax = 2,   // teacher top-K cache, pass 1
  kModeTopkCand = 3,  // teacher top-K cache, pass 2
  kModeDual = 4       // full-vocabulary loss: teacher then student logits of one tile
};

// Output staging: an epilogue warp writes its results 32 rows x 128 bytes at
// a time into its own shared-memory buffer (128-byte swizzle layout) and a
// TMA store (or reduce-add) moves the buffer to global memory, so the
// results leave the SM as whole lines instead of one 16-byte piece per row
// and thread.  The modes that write large outputs this way (pass 1: the
// stored exponentials; plain GEMMs: contiguous fp32 results) give one ring
// stage to the staging buffers.
constexpr int kStageWarpBytes = 32 * 128;
constexpr int kStagingBytes = kEpiWarps * kStageWarpBytes;

template <int MODE>
struct ModeCfg {
  static constexpr bool kStaged = MODE == kModePass1 || MODE == kModeStore || MODE == kModeDual;
  static constexpr int kStages = kStaged ? kMaxStages - 1 : kMaxStages;
  static constexpr size_t kSmem = 1024 + static_cast<size_t>(kStages) * kStageBytes +
                                  (kStaged ? kStagingBytes : 0) + sizeof(Ctl);
};
static_assert(ModeCfg<kModeStore>::kSmem <= 232448, "shared memory per CTA");
static_assert(ModeCfg<kModeDual>::kSmem <= 232448, "shared memory per CTA");

// Arrivals that complete one phase of the first CTA's barriers.
constexpr uint32_t kTemptyCount = 2 * kEpiWarps;          // epilogue warps of both CTAs
// first CTA: MMA, epilogue warps, B producer; second CTA: A and B producers, epilogue warps
constexpr uint32_t kSemptyCount = (1 + kEpiWarps + 1) + (2 + kEpiWarps);

// How a stage of an operand is loaded.
enum : int {
  kLoadK = 0,     // K-major: one 2-D box of 64 (K) x rows
  kLoadMN2d = 1,  // MN-major: one 2-D box of 64 (MN) x 64 (K) per 64-element atom
  kLoadMN3d = 2   // MN-major, atom-aligned: one 3-D box covering every atom
};

struct KParams {
  CUtensorMap tmA[2];
  CUtensorMap tmB[2];
  // staged outputs: kModeStore problem pi's result [M, N] fp32 (out_tma[pi] = 1:
  // stored, 2: added), kModePass1's stored exponentials [cpad, ldg] bf16 in
  // tmOut[0] (out_tma[0] = 1); 0: no staged output
  CUtensorMap tmOut[2];
  int out_tma[2];
  int a_mn[2], b_mn[2];
  int a_load[2], b_load[2];  // kLoadK / kLoadMN2d / kLoadMN3d
  int M[2], N[2], K[2];
  int bn[2];             // output tile width of the problem (multiple of 16, <= 256)
  uint32_t tx_bytes[2];  // bytes one pipeline stage receives in both CTAs together
  float* out[2];
  int64_t ldo[2];
  const float* row_scale[2];  // optional per-output-row factor (row m of the problem)
  int vec_ok[2];
  const int32_t* row_map[2];
  int64_t row_map_off[2];
  int accumulate[2];
  int count_mode[2];
  int nprob;
  const int32_t* n_valid;
  int64_t row0;
  int chunk;
  uint32_t* counter;
  uint32_t* err;
  uint64_t wait_limit_ns;  // 0: the default limit
  int withhold_arrival;    // test of the bounded waits: never announce stage 0's bytes
  const uint32_t* gate;    // when set and *gate == 0, the launch has no work
  // pass-1 epilogue
  float k2;
  int V;
  int64_t cpad;
  int n_pb;
  int K_top;
  const int32_t* rows;
  const int32_t* idx_sorted;
  const float* p_sorted;
  const uint16_t* boff;
  float* part_m;
  float* part_l;
  float* part_ps;
  uint16_t* u;
  int64_t ldg;
  const float* mref;     // [cpad] row references (nullptr: each block its own maximum)
  int32_t* row_flag;     // [cpad] set when a block of the row keeps its own maximum
  // top-K cache epilogues (rows are the chunk's positions, columns the vocabulary)
  uint64_t* bkey;        // [count][bkey_ld] largest rank key of each 128-column block
  int64_t bkey_ld;
  const uint64_t* tau;   // [count] the row's candidate threshold
  uint32_t* cnt;         // [count] candidates appended so far
  uint64_t* cand;        // [count][cap] candidate rank keys
  int64_t cap;
  // full-vocabulary loss (kModeDual): problem 0 is the teacher, problem 1 the
  // student; student statistics go to part_m / part_l and u
  uint16_t* u_t;         // [cpad, ldg] teacher exponentials 2^(t2 - m_t), bf16
  float* part_mt;        // [n_pb][cpad] teacher block max of t2
  float* part_lt;        // [n_pb][cpad] teacher block sum of 2^(t2 - m_t)
  float* part_a;         // [n_pb][cpad] block sum of 2^(t2 - m_t) (t2 - s2)
};

struct Sizes {
  int M[2], N[2], nkb[2], mt[2], nt[2], tiles[2], bn[2], b3d[2];
  int total;
  int count;
  int group_m;  // plain GEMMs: tile rows per raster group (0: row order)
};

__device__ __forceinline__ Sizes get_sizes(const KParams& P) {
  Sizes s;
  s.group_m = P.nprob == 1 ? 8 : 0;
  int count = P.chunk;
  if (P.n_valid != nullptr) {
    const long long c = static_cast<long long>(*P.n_valid) - P.row0;
    count = c < 0 ? 0 : (c > P.chunk ? P.chunk : static_cast<int>(c));
  }
  s.count = count;
  s.total = 0;
  if (P.gate != nullptr && *P.gate == 0u) return s;
#pragma unroll
  for (int pi = 0; pi < 2; ++pi) {
    int M = P.M[pi], N = P.N[pi], K = P.K[pi];
    if (P.count_mode[pi] == 1) M = min(M, count);
    if (P.count_mode[pi] == 2) K = min(K, count);
    s.M[pi] = M;
    s.N[pi] = N;
    s.nkb[pi] = (K + kBK - 1) / kBK;
    s.mt[pi] = (M + kPairM - 1) / kPairM;
    s.bn[pi] = P.bn[pi];
    s.b3d[pi] = P.b_load[pi] == kLoadMN3d;
    s.nt[pi] = s.bn[pi] > 0 ? (N + s.bn[pi] - 1) / s.bn[pi] : 0;
    int tiles = s.mt[pi] * s.nt[pi];
    if (pi >= P.nprob) tiles = 0;
    // Nothing to add: an accumulating problem with an empty reduction.
    if (s.nkb[pi] == 0 && P.accumulate[pi]) tiles = 0;
    s.tiles[pi] = tiles;
    s.total += tiles;
  }
  if (P.u_t != nullptr) {  // full-vocabulary pass: one tile covers both problems
    s.total = s.tiles[0];
    s.tiles[1] = 0;
  }
  return s;
}

struct Tile {
  int prob, m, n, nkb;
  int n_cols;  // MMA width of this tile: bn, or less for the last column tile
};

// Pass 1 walks the vocabulary slowly (m fastest) so that the CTAs running at
// the same time share one W tile; the backward walks the output columns
// fastest so that the CTAs running together share one A (G) slab.  A plain
// GEMM (one problem) goes through its output in groups of 8 tile rows, m
// fastest within a group, so that the tiles running together share both
// operands' tiles in L2 (measured at 8192^3: 1543-1555 against 1473-1479
// TFLOP/s with plain row order).
template <int MODE>
__device__ __forceinline__ Tile decode_tile(const Sizes& S, int t) {
  Tile tl;
  tl.prob = 0;
  if (t >= S.tiles[0]) {
    tl.prob = 1;
    t -= S.tiles[0];
  }
  const int pi = tl.prob;
  if (MODE == kModePass1 || MODE == kModeTopkMax || MODE == kModeTopkCand || MODE == kModeDual) {
    tl.m = t % S.mt[pi];
    tl.n = t / S.mt[pi];
  } else if (S.group_m > 0 && S.mt[pi] > S.group_m) {
    const int per = S.group_m * S.nt[pi];
    const int m0 = (t / per) * S.group_m;
    const int r = t % per;
    const int gsz = min(S.group_m, S.mt[pi] - m0);
    tl.m = m0 + r % gsz;
    tl.n = r / gsz;
  } else {
    tl.n = t % S.nt[pi];
    tl.m = t / S.nt[pi];
  }
  tl.nkb = S.nkb[pi] + (MODE == kModeDual ? S.nkb[1] : 0);
  // The pair MMA takes B as two halves of n_cols / 2 columns, one from each
  // CTA; a 3-D loaded B half must start on a 64-column atom (n_cols a
  // multiple of 128), any other B half on 8 columns (n_cols a multiple of 16).
  const int n_rest = S.N[pi] - tl.n * S.bn[pi];
  const int gran = S.b3d[pi] ? 128 : 16;
  tl.n_cols = min(S.bn[pi], (n_rest + gran - 1) / gran * gran);
  return tl;
}

__device__ __forceinline__ uint8_t* align_smem(uint8_t* raw) {
  const uint32_t a = smem_u32(raw);
  return raw + (((a + 1023u) & ~1023u) - a);
}

// Takes the next tile number from the shared ring (all lanes of the calling
// warp, or a single thread).  Returns false when the CTA has to stop.
__device__ __forceinline__ bool sched_pop(Ctl* ctl, int& slot, uint32_t& sphase, int& t,
                                          const WaitCtx& wc) {
  if (!mbar_wait(&ctl->sfull[slot], sphase, wc)) return false;
  t = *reinterpret_cast<volatile int*>(&ctl->sched_tile[slot]);
  return true;
}

// Hands the next tile number to the consumers of ring slot `slot` (first
// CTA's producer only): writes it into both CTAs' rings and arrives on both
// CTAs' "full" barriers of that slot.
__device__ __forceinline__ void sched_push(Ctl* ctl, int slot, int t) {
  const uint32_t tile_local = smem_u32(&ctl->sched_tile[slot]);
  const uint32_t bar_local = smem_u32(&ctl->sfull[slot]);
  st_cluster_u32(mapa_shared(tile_local, 0), static_cast<uint32_t>(t));
  st_cluster_u32(mapa_shared(tile_local, 1), static_cast<uint32_t>(t));
  mbar_arrive_cluster(mapa_shared(bar_local, 0));
  mbar_arrive_cluster(mapa_shared(bar_local, 1));
}

// Tells the first CTA that this role has taken ring slot `slot`.
__device__ __forceinline__ void sched_release(Ctl* ctl, int slot) {
  mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->sempty[slot]), 0));
}

// Loads this CTA's part of one operand for K block k0 into `dst`.
__device__ __forceinline__ void load_operand(uint8_t* dst, const CUtensorMap* m, int mode,
                                             uint32_t fb, int mn0, int mn_count, int k0) {
  if (mode == kLoadK) {
    tma_load_2d_pair(dst, m, fb, k0, mn0);
  } else if (mode == kLoadMN3d) {
    tma_load_3d_pair(dst, m, fb, 0, k0, mn0 / 64);
  } else {
    for (int a = 0; a < (mn_count + 63) / 64; ++a)
      tma_load_2d_pair(dst + a * kAtomBytes, m, fb, mn0 + a * 64, k0);
  }
}

// TMA producer of operand A (OPERAND = 0, warp 0) or B (OPERAND = 1, warp 10).
// The first CTA's A producer also runs the tile ring: it takes tile numbers
// from the global counter and pushes them to every role of both CTAs.
template <int MODE, int OPERAND>
__device__ void producer_loop(const KParams& P, const Sizes& S, uint8_t* smem, Ctl* ctl,
                              const WaitCtx& wc, uint32_t rank) {
  int stage = 0;
  uint32_t phase = 0;
  int slot = 0;
  uint32_t sphase = 0;
  bool aborted = false;
  bool first_tile = true;
  const bool ring_head = (OPERAND == 0) && rank == 0;
  while (true) {
    int t;
    if (ring_head) {
      if (!mbar_wait(&ctl->sempty[slot], sphase ^ 1u, wc)) {
        aborted = true;
        break;
      }
      t = static_cast<int>(atomicAdd(P.counter, 1u));
      if (t >= S.total) t = -1;
      sched_push(ctl, slot, t);
    } else {
      if (!sched_pop(ctl, slot, sphase, t, wc)) {
        aborted = true;
        break;
      }
      sched_release(ctl, slot);
    }
    if (++slot == kSched) {
      slot = 0;
      sphase ^= 1u;
    }
    if (t < 0) break;
    const Tile tl = decode_tile<MODE>(S, t);
    const int pi = tl.prob;
    // kModeDual: the first nkb[0] K blocks are the teacher's, then the student's
    const int nkb0 = MODE == kModeDual ? S.nkb[0] : tl.nkb;
    int mn0, mn_count;
    if (OPERAND == 0) {
      mn0 = tl.m * kPairM + static_cast<int>(rank) * kBM;
      mn_count = kBM;
    } else {
      // boxes cover the problem's half tile; this tile's halves may be narrower
      mn_count = S.bn[pi] >> 1;
      mn0 = tl.n * S.bn[pi] + static_cast<int>(rank) * (tl.n_cols >> 1);
    }
    const uint32_t tx = P.tx_bytes[pi];
    for (int kb = 0; kb < tl.nkb; ++kb) {
      if (!mbar_wait_fast(&ctl->empty[stage], phase ^ 1u, wc)) {
        aborted = true;
        break;
      }
      // Both CTAs' copies of A and B complete on the first CTA's barrier,
      // which expects the bytes of all four.
      if (OPERAND == 0 && rank == 0 && !(P.withhold_arrival && kb == 0 && first_tile))
        mbar_arrive_expect_tx(&ctl->full[stage], kb < nkb0 ? tx : P.tx_bytes[1]);
      const uint32_t fb = mapa_shared(smem_u32(&ctl->full[stage]), 0);
      uint8_t* dst = smem + stage * kStageBytes + (OPERAND == 0 ? 0 : kABytes);
      const int pk = kb < nkb0 ? pi : 1;
      const CUtensorMap* m = OPERAND == 0 ? &P.tmA[pk] : &P.tmB[pk];
      const int mode = OPERAND == 0 ? P.a_load[pk] : P.b_load[pk];
      load_operand(dst, m, mode, fb, mn0, mn_count, (kb < nkb0 ? kb : kb - nkb0) * kBK);
      if (++stage == ModeCfg<MODE>::kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    first_tile = false;
    if (aborted) break;
  }
  if (aborted) {
    // Let copies already issued land before the CTA's shared memory goes
    // away.  Their completion is counted in the first CTA's barriers, which
    // the other roles may no longer be waiting on, so wait a fixed 20 ms (a
    // copy takes microseconds).
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 20000000ull) {
    }
  }
}

// Pair MMA issue (first CTA, one thread).
template <int MODE>
__device__ void mma_loop(const KParams& P, const Sizes& S, uint8_t* smem, Ctl* ctl, uint32_t tmem,
                         const WaitCtx& wc) {
  int stage = 0;
  uint32_t phase = 0;
  int slot = 0;
  uint32_t sphase = 0;
  int it = 0;
  while (true) {
    int t;
    if (!sched_pop(ctl, slot, sphase, t, wc)) break;
    sched_release(ctl, slot);
    if (++slot == kSched) {
      slot = 0;
      sphase ^= 1u;
    }
    if (t < 0) break;
    const Tile tl = decode_tile<MODE>(S, t);
    // kModeDual: the teacher's accumulator is TMEM columns 0-255 (barriers
    // tfull/tempty[0]) and the student's 256-511 (barriers [1]); the epilogue
    // frees the teacher's as soon as it has copied it, so the next tile's
    // teacher product overlaps the epilogue.  Otherwise: two 256-column
    // accumulators used in turn.
    const int b = MODE == kModeDual ? 0 : (it & 1);
    const uint32_t tp = MODE == kModeDual ? (static_cast<uint32_t>(it) & 1u)
                                          : ((static_cast<uint32_t>(it) >> 1) & 1u);
    ++it;
    if (!mbar_wait(&ctl->tempty[b], tp ^ 1u, wc)) break;
    tc_fence_after();
    const uint32_t d_tmem0 = tmem + static_cast<uint32_t>(b * kBN);
    const int nkb0 = MODE == kModeDual ? S.nkb[0] : tl.nkb;
    const int pi = tl.prob;
    const int a_mn = P.a_mn[pi], b_mn = P.b_mn[pi];
    const uint32_t idesc = idesc_bf16_f32(kPairM, tl.n_cols, a_mn, b_mn);
    bool ok = true;
    for (int kb = 0; kb < tl.nkb; ++kb) {
      if (MODE == kModeDual && kb == nkb0) {
        // teacher product done; the student's accumulator must be free
        umma_commit_pair_both(&ctl->tfull[0]);
        if (!mbar_wait(&ctl->tempty[1], tp ^ 1u, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      if (!mbar_wait_fast(&ctl->full[stage], phase, wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sa = smem_u32(smem + stage * kStageBytes);
      const uint32_t sb = sa + kABytes;
      const bool second = kb >= nkb0;  // kModeDual: the student's K blocks
      const uint32_t d_tmem = d_tmem0 + (second ? static_cast<uint32_t>(kBN) : 0u);
      const int kb_in = second ? kb - nkb0 : kb;
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk) {
        // K-major: the next 16 K elements are 32 bytes further along each
        // 128-byte row.  MN-major: they are the next 16 rows of 128 bytes.
        const uint64_t ad = a_mn ? sdesc_sw128(sa + kk * 2048, kAtomBytes, 1024)
                                 : sdesc_sw128(sa + kk * 32, 16, 1024);
        const uint64_t bd = b_mn ? sdesc_sw128(sb + kk * 2048, kAtomBytes, 1024)
                                 : sdesc_sw128(sb + kk * 32, 16, 1024);
        umma_bf16_pair(d_tmem, ad, bd, idesc, (kb_in > 0 || kk > 0) ? 1u : 0u);
      }
      umma_commit_pair_both(&ctl->empty[stage]);
      if (++stage == ModeCfg<MODE>::kStages) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (!ok) break;
    umma_commit_pair_both(&ctl->tfull[MODE == kModeDual ? 1 : b]);
  }
  // Every MMA this thread issued must finish before TMEM is freed.
  umma_commit_pair_local(&ctl->drain);
  mbar_wait_drain(&ctl->drain, 0, P.err);
}

// ------------------------------------------------------------------ epilogues

__device__ __forceinline__ void load_acc128(uint32_t ta, float (&v0)[32], float (&v1)[32],
                                            float (&v2)[32], float (&v3)[32]) {
  tmem_ld_x32(ta, v0);
  tmem_ld_x32(ta + 32, v1);
  tmem_ld_x32(ta + 64, v2);
  tmem_ld_x32(ta + 96, v3);
  tmem_ld_wait();
  reg_fence(v0);
  reg_fence(v1);
  reg_fence(v2);
  reg_fence(v3);
}

__device__ __forceinline__ void store_chunk32(float* dst, const float (&v)[32], int nc, bool vec,
                                              bool acc) {
  if (vec && nc >= 32) {
    float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float4 x = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      if (acc) {
        const float4 o = d4[j];
        x.x += o.x;
        x.y += o.y;
        x.z += o.z;
        x.w += o.w;
      }
      d4[j] = x;
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j < nc) dst[j] = acc ? dst[j] + v[j] : v[j];
    }
  }
}

// One 16-byte piece (piece c of 8) of this lane's 128-byte row of a staging
// buffer, at its place in the 128-byte swizzle layout.
__device__ __forceinline__ void stage_put(uint8_t* buf, int lane, int c, uint32_t w0, uint32_t w1,
                                          uint32_t w2, uint32_t w3) {
  const uint32_t row = smem_u32(buf) + static_cast<uint32_t>(lane) * 128u;
  st_shared_v4(row + ((static_cast<uint32_t>(c) ^ (static_cast<uint32_t>(lane) & 7u)) << 4), w0,
               w1, w2, w3);
}

// Sends the warp's filled staging buffer (32 rows of 128 bytes) to global
// memory as one box at (x, y), and waits until the buffer may be reused.
__device__ __forceinline__ void stage_flush(const CUtensorMap* m, uint8_t* buf, int lane, int x,
                                            int y, bool add) {
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    // streamed outputs: evict-first in L2, so that they leave room for the
    // operands (measured: pass 1 reads 2.95 instead of 3.44 GB of W per
    // 8192-token chunk)
    const uint64_t pol = l2_evict_first_policy();
    if (add) tma_reduce_add_2d(m, buf, x, y, pol);
    else tma_store_2d(m, buf, x, y, pol);
    bulk_commit_group();
    bulk_wait_group_read0();
  }
  __syncwarp();
}

// Writes one piece of 32 rows x 128 bytes, held one row per lane as 32 words,
// into the warp's staging buffer in the 128-byte swizzle layout of the
// output's tensor map, then lane 0 stores it (or adds it) at (x, y) with TMA
// and waits until the buffer has been read, so the next piece may reuse it.
// The rows and columns of the box that fall outside the tensor are dropped
// by the TMA unit.
__device__ __forceinline__ void stage_piece(const CUtensorMap* m, uint8_t* buf,
                                            const uint32_t (&w)[32], int lane, int x, int y,
                                            bool add) {
  const uint32_t row = smem_u32(buf) + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
  for (int c = 0; c < 8; ++c)
    st_shared_v4(row + ((static_cast<uint32_t>(c) ^ (static_cast<uint32_t>(lane) & 7u)) << 4),
                 w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
  stage_flush(m, buf, lane, x, y, add);
}

__device__ __forceinline__ void stage_f32(const CUtensorMap* m, uint8_t* buf, const float (&v)[32],
                                          int lane, int x, int y, bool add) {
  const uint32_t (&w)[32] = *reinterpret_cast<const uint32_t(*)[32]>(v);
  stage_piece(m, buf, w, lane, x, y, add);
}

__device__ void epilogue_store(const KParams& P, const Sizes& S, Ctl* ctl, uint32_t tmem,
                               const WaitCtx& wc, int warp, int lane, int rank, uint8_t* wbuf) {
  const int q = warp & 3;           // TMEM lane quarter this warp may read
  const int half = (warp - 2) >> 2; // which 128 columns of the 256
  int slot = 0;
  uint32_t sphase = 0;
  int it = 0;
  while (true) {
    int t = -1;
    bool ok = sched_pop(ctl, slot, sphase, t, wc);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    __syncwarp();
    if (lane == 0) sched_release(ctl, slot);
    if (++slot == kSched) {
      slot = 0;
      sphase ^= 1u;
    }
    if (t < 0) break;
    const Tile tl = decode_tile<kModeStore>(S, t);
    const int b = it & 1;
    const uint32_t tp = (static_cast<uint32_t>(it) >> 1) & 1u;
    ++it;
    ok = mbar_wait(&ctl->tfull[b], tp, wc);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    tc_fence_after();
    const int pi = tl.prob;
    float v0[32], v1[32], v2[32], v3[32];
    if (tl.nkb > 0) {
      const uint32_t ta = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                          static_cast<uint32_t>(b * kBN + half * 128);
      load_acc128(ta, v0, v1, v2, v3);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) v0[j] = v1[j] = v2[j] = v3[j] = 0.f;
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->tempty[b]), 0));

    const int i0 = tl.m * kPairM + rank * kBM + q * 32;  // the warp's first row
    const int i = i0 + lane;
    const int col0 = tl.n * S.bn[pi] + half * 128;
    const int ncols = min(S.bn[pi] - half * 128, S.N[pi] - col0);  // columns of this half
    if (P.out_tma[pi] != 0) {
      // contiguous fp32 result: staged, whole-line TMA stores (or adds)
      if (i0 < S.M[pi] && ncols > 0) {
        const bool add = P.out_tma[pi] == 2;
        stage_f32(&P.tmOut[pi], wbuf, v0, lane, col0, i0, add);
        if (ncols > 32) stage_f32(&P.tmOut[pi], wbuf, v1, lane, col0 + 32, i0, add);
        if (ncols > 64) stage_f32(&P.tmOut[pi], wbuf, v2, lane, col0 + 64, i0, add);
        if (ncols > 96) stage_f32(&P.tmOut[pi], wbuf, v3, lane, col0 + 96, i0, add);
      }
    } else if (i < S.M[pi] && ncols > 0) {
      if (P.row_scale[pi] != nullptr) {
        const float f = P.row_scale[pi][i];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          v0[j] *= f;
          v1[j] *= f;
          v2[j] *= f;
          v3[j] *= f;
        }
      }
      const int64_t orow =
          P.row_map[pi] != nullptr ? P.row_map[pi][P.row_map_off[pi] + i] : static_cast<int64_t>(i);
      float* dst = P.out[pi] + orow * P.ldo[pi] + col0;
      const int nc = min(128, ncols);
      const bool vec = P.vec_ok[pi] != 0;
      const bool acc = P.accumulate[pi] != 0;
      store_chunk32(dst, v0, nc, vec, acc);
      if (nc > 32) store_chunk32(dst + 32, v1, nc - 32, vec, acc);
      if (nc > 64) store_chunk32(dst + 64, v2, nc - 64, vec, acc);
      if (nc > 96) store_chunk32(dst + 96, v3, nc - 96, vec, acc);
    }
  }
  // every staged store complete before the kernel ends
  if (lane == 0) bulk_wait_group0();
  __syncwarp();
}

// Logsumexp statistics of 32 consecutive logits of one row, in base-2 units
// s2 = z * k2 relative to the block's reference m2: the sum of the
// exponentials into l, and the exponentials themselves as 16 words of two
// bf16 (lower column in the low half) into w, for the staged store.
template <bool kMasked>
__device__ __forceinline__ void lse_chunk32(const float (&v)[32], int nvalid, float k2, float m2,
                                            float& l, uint32_t* w) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    float e0 = ex2_approx(fmaf(v[2 * j], k2, -m2));
    float e1 = ex2_approx(fmaf(v[2 * j + 1], k2, -m2));
    if (kMasked) {
      e0 = (2 * j < nvalid) ? e0 : 0.f;
      e1 = (2 * j + 1 < nvalid) ? e1 : 0.f;
    }
    l += e0 + e1;
    w[j] = pack_bf16x2(e0, e1);
  }
}

__device__ __forceinline__ float max32(const float (&v)[32], int nvalid, bool masked) {
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    if (!masked || j < nvalid) m = fmaxf(m, v[j]);
  }
  return m;
}

__device__ void epilogue_pass1(const KParams& P, const Sizes& S, Ctl* ctl, uint32_t tmem,
                               const WaitCtx& wc, int warp, int lane, int rank, uint8_t* wbuf) {
  const int q = warp & 3;
  const int half = (warp - 2) >> 2;
  int slot = 0;
  uint32_t sphase = 0;
  int it = 0;
  const float k2 = P.k2;
  while (true) {
    int t = -1;
    bool ok = sched_pop(ctl, slot, sphase, t, wc);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    __syncwarp();
    if (lane == 0) sched_release(ctl, slot);
    if (++slot == kSched) {
      slot = 0;
      sphase ^= 1u;
    }
    if (t < 0) break;
    const Tile tl = decode_tile<kModePass1>(S, t);
    const int b = it & 1;
    const uint32_t tp = (static_cast<uint32_t>(it) >> 1) & 1u;
    ++it;

    const int i0 = tl.m * kPairM + rank * kBM + q * 32;      // the warp's first row
    const int i = i0 + lane;                                   // row within the chunk
    const int col0 = tl.n * kBN + half * 128;  // first vocabulary column of this block
    const int pb = tl.n * 2 + half;            // 128-column block index
    const bool block_live = pb < P.n_pb;       // the same for the whole warp
    const bool live = (i < S.count) && block_live;
    // Teacher entries of this row that fall in this column block.
    int lo = 0, hi = 0;
    const int32_t* lidx = nullptr;
    const float* lp = nullptr;
    float mr = 0.f;  // the row's reference (loaded before the accumulator wait)
    if (live) {
      lo = P.boff[static_cast<int64_t>(pb) * P.cpad + i];
      hi = P.boff[static_cast<int64_t>(pb + 1) * P.cpad + i];
      const int64_t r = P.rows[P.row0 + i];
      lidx = P.idx_sorted + r * P.K_top;
      lp = P.p_sorted + r * P.K_top;
      if (P.mref != nullptr) mr = P.mref[i];
    }

    ok = mbar_wait(&ctl->tfull[b], tp, wc);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    tc_fence_after();
    const uint32_t ta = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                        static_cast<uint32_t>(b * kBN + half * 128);
    float v0[32], v1[32], v2[32], v3[32];
    load_acc128(ta, v0, v1, v2, v3);

    // Logits at the teacher's indices: the warp walks its lanes' pending
    // entries one at a time, each a single-column TMEM load.
    float ps = 0.f;
    uint32_t pend = __ballot_sync(0xffffffffu, lo < hi);
    while (pend != 0u) {
      const int src = __ffs(pend) - 1;
      int jj = 0;
      if (lo < hi) jj = lidx[lo] - col0;
      const int j = __shfl_sync(0xffffffffu, jj, src) & 127;
      float z = tmem_ld_x1(ta + static_cast<uint32_t>(j));
      tmem_ld_wait();
      reg_fence1(z);
      if (lane == src) {
        ps = fmaf(lp[lo], z, ps);
        ++lo;
      }
      pend = __ballot_sync(0xffffffffu, lo < hi);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->tempty[b]), 0));

    // Every lane of a live block computes its row's exponentials (rows past
    // the chunk's count hold values nobody reads: they are stored with the
    // rest of the box, and cleared or ignored later); the statistics and the
    // row flag are written for the chunk's rows only.
    if (block_live && i0 < S.count) {
      const int nv = min(128, P.V - col0);
      float l = 0.f;
      float m2;
      // The block's exponentials are taken relative to the row's reference
      // when its maximum is at most kRefSlack above it (then every block of
      // the row shares one reference and the gradient products can use the
      // stored values directly), else relative to its own maximum.
      uint32_t wa[32], wb[32];  // columns 0-63 and 64-127, two bf16 per word
      if (nv == 128) {
        const float mx = fmaxf(fmaxf(max32(v0, 32, false), max32(v1, 32, false)),
                               fmaxf(max32(v2, 32, false), max32(v3, 32, false)));
        m2 = mx * k2;
        if (live && P.mref != nullptr) {
          if (m2 - mr <= kRefSlack) m2 = mr;
          else P.row_flag[i] = 1;
        }
        lse_chunk32<false>(v0, 32, k2, m2, l, wa);
        lse_chunk32<false>(v1, 32, k2, m2, l, wa + 16);
        lse_chunk32<false>(v2, 32, k2, m2, l, wb);
        lse_chunk32<false>(v3, 32, k2, m2, l, wb + 16);
      } else {
        const float mx = fmaxf(fmaxf(max32(v0, nv, true), max32(v1, nv - 32, true)),
                               fmaxf(max32(v2, nv - 64, true), max32(v3, nv - 96, true)));
        m2 = mx * k2;
        if (live && P.mref != nullptr) {
          if (m2 - mr <= kRefSlack) m2 = mr;
          else P.row_flag[i] = 1;
        }
        lse_chunk32<true>(v0, nv, k2, m2, l, wa);
        lse_chunk32<true>(v1, nv - 32, k2, m2, l, wa + 16);
        lse_chunk32<true>(v2, nv - 64, k2, m2, l, wb);
        lse_chunk32<true>(v3, nv - 96, k2, m2, l, wb + 16);
      }
      if (P.out_tma[0] != 0) {  // the stored exponentials, through the staging buffer
        stage_piece(&P.tmOut[0], wbuf, wa, lane, col0, i0, false);
        stage_piece(&P.tmOut[0], wbuf, wb, lane, col0 + 64, i0, false);
      }
      if (live) {
        const int64_t o = static_cast<int64_t>(pb) * P.cpad + i;
        P.part_m[o] = m2;
        P.part_l[o] = l;
        P.part_ps[o] = ps * k2;
      }
    }
  }
  if (lane == 0) bulk_wait_group0();
  __syncwarp();
}

// Rank key of logit z at vocabulary index v: a larger key ranks first.  The
// high word orders the float (NaN lowest, -0 folded into +0), the low word
// puts the lower index first among equal logits.
__device__ __forceinline__ uint64_t rank_key(float z, uint32_t v) {
  uint32_t u = __float_as_uint(z);
  if (z == 0.0f) u = 0u;
  uint32_t o = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  if (z != z) o = 0u;
  return (static_cast<uint64_t>(o) << 32) | static_cast<uint64_t>(0xFFFFFFFFu - v);
}

template <int N>
__device__ __forceinline__ uint64_t max_key32(const float (&v)[N], int col, int nvalid,
                                              uint64_t best) {
#pragma unroll
  for (int j = 0; j < N; ++j) {
    if (j < nvalid) {
      const uint64_t k = rank_key(v[j], static_cast<uint32_t>(col + j));
      best = k > best ? k : best;
    }
  }
  return best;
}

// The block maximum as in max_key32, and every key >= tau appended to the
// row's candidate list (slots past the capacity are counted, not written).
__device__ __forceinline__ uint64_t max_append32(const float (&v)[32], int col, int nvalid,
                                                 uint64_t best, uint64_t tau, uint32_t* cnt,
                                                 uint64_t* cand, int64_t cap) {
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    if (j < nvalid) {
      const uint64_t k = rank_key(v[j], static_cast<uint32_t>(col + j));
      best = k > best ? k : best;
      if (k >= tau) {
        const uint32_t slot = atomicAdd(cnt, 1u);
        if (slot < cap) cand[slot] = k;
      }
    }
  }
  return best;
}

// Top-K cache epilogues.  Each thread owns one row and one 128-column block
// of the tile.
//   kModeTopkMax:  the block's largest rank key -> bkey[row][block];
//   kModeTopkCand: the same, and every key >= the row's threshold tau is
//                  appended to the row's candidates (the count goes on past
//                  the capacity, so an overflowing row is recognisable).
template <int MODE>
__device__ void epilogue_topk(const KParams& P, const Sizes& S, Ctl* ctl, uint32_t tmem,
                              const WaitCtx& wc, int warp, int lane, int rank) {
  const int q = warp & 3;
  const int half = (warp - 2) >> 2;
  int slot = 0;
  uint32_t sphase = 0;
  int it = 0;
  while (true) {
    int t = -1;
    bool ok = sched_pop(ctl, slot, sphase, t, wc);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    __syncwarp();
    if (lane == 0) sched_release(ctl, slot);
    if (++slot == kSched) {
      slot = 0;
      sphase ^= 1u;
    }
    if (t < 0) break;
    const Tile tl = decode_tile<MODE>(S, t);
    const int b = it & 1;
    const uint32_t tp = (static_cast<uint32_t>(it) >> 1) & 1u;
    ++it;
    const int i = tl.m * kPairM + rank * kBM + q * 32 + lane;  // row of the chunk
    const int col0 = tl.n * kBN + half * 128;
    const int pb = tl.n * 2 + half;
    const bool live = (i < S.count) && (pb < P.n_pb);
    uint64_t tau = 0;
    if (MODE == kModeTopkCand && live) tau = P.tau[i];
    ok = mbar_wait(&ctl->tfull[b], tp, wc);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    tc_fence_after();
    const uint32_t ta = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                        static_cast<uint32_t>(b * kBN + half * 128);
    float v0[32], v1[32], v2[32], v3[32];
    load_acc128(ta, v0, v1, v2, v3);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->tempty[b]), 0));
    if (!live) continue;
    const int nv = min(128, P.V - col0);
    uint64_t best = 0;
    if (MODE == kModeTopkMax) {
      best = max_key32(v0, col0, nv, best);
      best = max_key32(v1, col0 + 32, nv - 32, best);
      best = max_key32(v2, col0 + 64, nv - 64, best);
      best = max_key32(v3, col0 + 96, nv - 96, best);
    } else {
      uint32_t* cnt = P.cnt + i;
      uint64_t* cand = P.cand + static_cast<int64_t>(i) * P.cap;
      best = max_append32(v0, col0, nv, best, tau, cnt, cand, P.cap);
      best = max_append32(v1, col0 + 32, nv - 32, best, tau, cnt, cand, P.cap);
      best = max_append32(v2, col0 + 64, nv - 64, best, tau, cnt, cand, P.cap);
      best = max_append32(v3, col0 + 96, nv - 96, best, tau, cnt, cand, P.cap);
    }
    P.bkey[static_cast<int64_t>(i) * P.bkey_ld + pb] = best;
  }
}

// Full-vocabulary loss: maximum of up to 16 student logits (raw z) from TMEM.
__device__ __forceinline__ float max16_tmem(uint32_t ta, int nvalid, float m) {
  float s[16];
  tmem_ld_x16(ta, s);
  tmem_ld_wait();
  reg_fence(s);
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if (j < nvalid) m = fmaxf(m, s[j]);
  return m;
}

// Full-vocabulary loss epilogue.  The tile's teacher logits are in TMEM
// columns 0-255 and the student's in 256-511; each thread owns one row and
// one 128-column block, each warp 32 rows of it.  In two phases:
//  1. the warp copies its 128 teacher logits per row into registers and frees
//     the teacher accumulator at once (the next tile's teacher product then
//     runs during the rest of this epilogue); it takes the block maximum m_t,
//     and, while the student product is still running, the exponentials
//     2^(t2 - m_t) (t2 = z_t k2), their sum l_t, and stores them (bf16) through
//     the staging buffer, 64 columns per TMA store;
//  2. once the student product is done: the student's maximum m_s, its
//     exponentials (sum l_s, stored the same way) and the cross term
//     a = sum of 2^(t2 - m_t) (t2 - s2), which recomputes the teacher's
//     exponential rather than keep 128 more values in registers.
__device__ void epilogue_dual(const KParams& P, const Sizes& S, Ctl* ctl, uint32_t tmem,
                              const WaitCtx& wc, int warp, int lane, int rank, uint8_t* wbuf) {
  const int q = warp & 3;
  const int half = (warp - 2) >> 2;
  int slot = 0;
  uint32_t sphase = 0;
  int it = 0;
  const float k2 = P.k2;
  const uint32_t tempty0 = mapa_shared(smem_u32(&ctl->tempty[0]), 0);
  const uint32_t tempty1 = mapa_shared(smem_u32(&ctl->tempty[1]), 0);
  while (true) {
    int t = -1;
    bool ok = sched_pop(ctl, slot, sphase, t, wc);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    __syncwarp();
    if (lane == 0) sched_release(ctl, slot);
    if (++slot == kSched) {
      slot = 0;
      sphase ^= 1u;
    }
    if (t < 0) break;
    const Tile tl = decode_tile<kModeDual>(S, t);
    const uint32_t tp = static_cast<uint32_t>(it) & 1u;
    ++it;
    const int i0 = tl.m * kPairM + rank * kBM + q * 32;  // the warp's first row
    const int i = i0 + lane;
    const int col0 = tl.n * kBN + half * 128;
    const int pb = tl.n * 2 + half;
    const bool block_live = pb < P.n_pb;                  // warp-uniform
    const bool store = block_live && i0 < S.count;        // warp-uniform: the warp stores
    const bool live = block_live && i < S.count;          // this row's statistics
    const int nv = block_live ? min(128, P.V - col0) : 0;  // warp-uniform
    const uint32_t ta = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                        static_cast<uint32_t>(half * 128);
    const uint32_t ts = ta + static_cast<uint32_t>(kBN);
    // phase 1: teacher logits -> registers, then free the teacher accumulator
    ok = mbar_wait(&ctl->tfull[0], tp, wc);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    tc_fence_after();
    float tv[128];
    {
      float (&t0)[32] = *reinterpret_cast<float(*)[32]>(tv);
      float (&t1)[32] = *reinterpret_cast<float(*)[32]>(tv + 32);
      float (&t2)[32] = *reinterpret_cast<float(*)[32]>(tv + 64);
      float (&t3)[32] = *reinterpret_cast<float(*)[32]>(tv + 96);
      load_acc128(ta, t0, t1, t2, t3);
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive_cluster(tempty0);
    float mt = -INFINITY;
#pragma unroll
    for (int j = 0; j < 128; ++j)
      if (j < nv) mt = fmaxf(mt, tv[j]);
    const float mt2 = mt * k2;
    float lt = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {  // 64 columns per stored box
      if (nv > 64 * h) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // 8 columns per 16-byte piece
          uint32_t w[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int c0 = 64 * h + 8 * c + 2 * j;
            // the same expression as the cross term's below
            const float e0 = c0 < nv ? ex2_approx(tv[c0] * k2 - mt2) : 0.f;
            const float e1 = c0 + 1 < nv ? ex2_approx(tv[c0 + 1] * k2 - mt2) : 0.f;
            lt += e0 + e1;
            w[j] = pack_bf16x2(e0, e1);
          }
          if (store) stage_put(wbuf, lane, c, w[0], w[1], w[2], w[3]);
        }
        if (store) stage_flush(&P.tmOut[1], wbuf, lane, col0 + 64 * h, i0, false);
      }
    }
    // phase 2: student logits: maximum, then exponentials and the cross term
    ok = mbar_wait(&ctl->tfull[1], tp, wc);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) break;
    tc_fence_after();
    float ms = -INFINITY;
#pragma unroll
    for (int c = 0; c < 8; ++c)
      if (nv > 16 * c) ms = max16_tmem(ts + 16 * c, nv - 16 * c, ms);
    const float ms2 = ms * k2;
    float ls = 0.f, a = 0.f;
    // every lane takes part in the (warp-collective) TMEM loads
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (nv > 64 * h) {
#pragma unroll
        for (int c16 = 0; c16 < 4; ++c16) {
          const int cb = 64 * h + 16 * c16;  // first column of these 16
          float sv[16];
          if (nv > cb) {
            tmem_ld_x16(ts + cb, sv);
            tmem_ld_wait();
            reg_fence(sv);
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) sv[j] = 0.f;
          }
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              float es[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int c = cb + 8 * g + 2 * j + e;
                es[e] = 0.f;
                if (c < nv) {
                  const float t2 = tv[c] * k2, s2 = sv[8 * g + 2 * j + e] * k2;
                  es[e] = ex2_approx(s2 - ms2);
                  ls += es[e];
                  a = fmaf(ex2_approx(t2 - mt2), t2 - s2, a);
                }
              }
              w[j] = pack_bf16x2(es[0], es[1]);
            }
            if (store) stage_put(wbuf, lane, 2 * c16 + g, w[0], w[1], w[2], w[3]);
          }
        }
        if (store) stage_flush(&P.tmOut[0], wbuf, lane, col0 + 64 * h, i0, false);
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive_cluster(tempty1);
    if (live) {
      const int64_t o = static_cast<int64_t>(pb) * P.cpad + i;
      P.part_mt[o] = mt2;
      P.part_lt[o] = lt;
      P.part_a[o] = a;
      P.part_m[o] = ms2;
      P.part_l[o] = ls;
    }
  }
  // every staged store complete before the kernel ends
  if (lane == 0) bulk_wait_group0();
  __syncwarp();
}

template <int MODE>
__global__ void __launch_bounds__(kThreads, 1) tc_gemm_kernel(const __grid_constant__ KParams P) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem(smem_raw);
  uint8_t* staging = smem + ModeCfg<MODE>::kStages * kStageBytes;
  Ctl* ctl = reinterpret_cast<Ctl*>(staging + (ModeCfg<MODE>::kStaged ? kStagingBytes : 0));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  // Both CTAs of a pair see the same sizes, so both leave here or neither.
  const Sizes S = get_sizes(P);
  if (S.total == 0) return;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int s = 0; s < ModeCfg<MODE>::kStages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl->tfull[b], 1);
      mbar_init(&ctl->tempty[b], kTemptyCount);
    }
#pragma unroll
    for (int s = 0; s < kSched; ++s) {
      mbar_init(&ctl->sfull[s], 1);
      mbar_init(&ctl->sempty[s], kSemptyCount);
    }
    mbar_init(&ctl->drain, 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&P.tmA[0]);
    tma_prefetch_desc(&P.tmB[0]);
    if (P.nprob > 1) {
      tma_prefetch_desc(&P.tmA[1]);
      tma_prefetch_desc(&P.tmB[1]);
    }
  }
  // Both CTAs' barriers are initialised before either CTA arrives on the
  // other's, and the other CTA is running before the pair allocates TMEM.
  cluster_sync_all();
  if (warp == 1) tmem_alloc_pair(&ctl->tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const WaitCtx wc{&ctl->abort, mapa_shared(smem_u32(&ctl->abort), rank ^ 1u), P.err,
                   P.wait_limit_ns != 0 ? P.wait_limit_ns : kWaitLimitNs};

  if (warp == 0) {
    if (lane == 0) producer_loop<MODE, 0>(P, S, smem, ctl, wc, rank);
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) mma_loop<MODE>(P, S, smem, ctl, tmem, wc);
  } else if (warp == kBProducerWarp) {
    if (lane == 0) producer_loop<MODE, 1>(P, S, smem, ctl, wc, rank);
  } else {
    uint8_t* wbuf = staging + (warp - 2) * kStageWarpBytes;  // this warp's staging buffer
    if (MODE == kModePass1)
      epilogue_pass1(P, S, ctl, tmem, wc, warp, lane, static_cast<int>(rank), wbuf);
    else if (MODE == kModeStore)
      epilogue_store(P, S, ctl, tmem, wc, warp, lane, static_cast<int>(rank), wbuf);
    else if (MODE == kModeDual)
      epilogue_dual(P, S, ctl, tmem, wc, warp, lane, static_cast<int>(rank), wbuf);
    else
      epilogue_topk<MODE>(P, S, ctl, tmem, wc, warp, lane, static_cast<int>(rank));
  }

  // No CTA leaves while the other may still arrive on its barriers or have
  // pair MMAs read its shared memory; then the pair frees its TMEM together.
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

template <int MODE>
cudaError_t launch_mode(const KParams& P, int num_sms, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<MODE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(ModeCfg<MODE>::kSmem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof(cfg));
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = ModeCfg<MODE>::kSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // One pair per two SMs, as many as can be resident together (persistent).
  int pairs = num_sms / 2;
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  int fit = 0;
  if (cudaOccupancyMaxActiveClusters(&fit, tc_gemm_kernel<MODE>, &cfg) == cudaSuccess && fit > 0 &&
      fit < pairs)
    pairs = fit;
  cudaGetLastError();
  if (pairs < 1) pairs = 1;
  cfg.gridDim = dim3(2 * pairs, 1, 1);
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<MODE>, P);
}

// Output tile width for an N-wide output.  An MN-major B whose rows are whole
// 64-element atoms takes 256-wide tiles, so each CTA's half starts on an atom
// and loads with one 3-D box (the last tile multiplies only its real
// columns).  Otherwise: the fewest 256-wide tiles, then the narrowest multiple
// of 16 that still covers N with that many tiles (d = 2880 -> 12 tiles of 240
// instead of 11.25 tiles of 256).
int tile_width(int64_t N, int b_mn, int64_t b_inner) {
  if (b_mn && b_inner % 64 == 0) return kBN;
  const int64_t tiles = (N + kBN - 1) / kBN;
  const int64_t w = (N + tiles - 1) / tiles;
  return static_cast<int>((w + 15) / 16 * 16);
}

// Encodes the tensor map of one operand for the given load mode (see
// load_operand); rows_per_tile is this CTA's share of the tile along M or N.
bool encode_operand(CUtensorMap* m, const void* base, int mode, int64_t inner, int64_t outer,
                    int64_t ld, int rows_per_tile) {
  if (mode == kLoadK) return encode_tmap_bf16(m, base, inner, outer, ld, kBK, rows_per_tile);
  if (mode == kLoadMN3d)
    return encode_tmap_bf16_mn3d(m, base, inner, outer, ld, rows_per_tile / 64, kBK);
  return encode_tmap_bf16(m, base, inner, outer, ld, 64, kBK);
}

// Load mode of an operand: MN-major tiles use one 3-D box when the stored
// rows are whole atoms and every CTA's part starts on an atom (its share of
// the tile is a multiple of 64).
int load_mode(int mn, int64_t inner, int share) {
  if (!mn) return kLoadK;
  return (inner % 64 == 0 && share % 64 == 0) ? kLoadMN3d : kLoadMN2d;
}

uint32_t stage_bytes(int mode, int share) {
  if (mode == kLoadK) return static_cast<uint32_t>(share) * kBK * 2;
  return static_cast<uint32_t>((share + 63) / 64) * kAtomBytes;
}

}  // namespace

cudaError_t launch_tc_gemm(const TcGemmArgs& g, cudaStream_t s) {
  KParams P;
  memset(&P, 0, sizeof(P));
  for (int pi = 0; pi < g.nprob; ++pi) {
    const TcProblem& q = g.pr[pi];
    const int bn = tile_width(q.N, q.b_mn, q.b_inner);
    // each CTA: its 128 rows of A and its bn/2 columns of B
    const int a_load = load_mode(q.a_mn, q.a_inner, kBM);
    const int b_load = load_mode(q.b_mn, q.b_inner, bn / 2);
    if (!encode_operand(&P.tmA[pi], q.A, a_load, q.a_inner, q.a_outer, q.lda, kBM) ||
        !encode_operand(&P.tmB[pi], q.B, b_load, q.b_inner, q.b_outer, q.ldb, bn / 2))
      return cudaErrorInvalidValue;
    P.a_mn[pi] = q.a_mn;
    P.b_mn[pi] = q.b_mn;
    P.a_load[pi] = a_load;
    P.b_load[pi] = b_load;
    P.bn[pi] = bn;
    P.tx_bytes[pi] = 2u * (stage_bytes(a_load, kBM) + stage_bytes(b_load, bn / 2));
    P.M[pi] = static_cast<int>(q.M);
    P.N[pi] = static_cast<int>(q.N);
    P.K[pi] = static_cast<int>(q.K);
    P.out[pi] = q.out;
    P.ldo[pi] = q.ldo;
    P.vec_ok[pi] = (q.ldo % 4 == 0) && (reinterpret_cast<uintptr_t>(q.out) % 16 == 0);
    P.row_map[pi] = q.row_map;
    P.row_map_off[pi] = q.row_map_off;
    P.row_scale[pi] = q.row_scale;
    // a contiguous result (no row map, no row factor) leaves through the
    // staging buffers as whole-line TMA stores, or adds when accumulating
    if (q.row_map == nullptr && q.row_scale == nullptr && (q.ldo * 4) % 16 == 0 &&
        (reinterpret_cast<uintptr_t>(q.out) & 15u) == 0) {
      if (!encode_tmap_store(&P.tmOut[pi], q.out, true, q.N, q.M, q.ldo, 32, 32))
        return cudaErrorInvalidValue;
      P.out_tma[pi] = q.accumulate ? 2 : 1;
    }
    P.accumulate[pi] = q.accumulate;
    P.count_mode[pi] = q.count_mode;
  }
  if (g.nprob == 1) P.tmA[1] = P.tmA[0], P.tmB[1] = P.tmB[0];
  P.nprob = g.nprob;
  P.n_valid = g.n_valid;
  P.row0 = g.row0;
  P.chunk = g.chunk;
  P.counter = g.counter;
  P.err = g.err;
  P.wait_limit_ns = g.wait_limit_ns;
  P.withhold_arrival = g.withhold_arrival;
  cudaError_t e = cudaMemsetAsync(g.counter, 0, sizeof(uint32_t), s);
  if (e != cudaSuccess) return e;
  return launch_mode<kModeStore>(P, g.num_sms, s);
}

cudaError_t launch_tc_pass1(const Pass1Args& p, const ChunkArgs& a, cudaStream_t s) {
  KParams P;
  memset(&P, 0, sizeof(P));
  if (!encode_operand(&P.tmA[0], p.hc, kLoadK, p.d, a.cpad, p.d, kBM) ||
      !encode_operand(&P.tmB[0], p.W, kLoadK, p.d, a.V, p.d, kBN / 2))
    return cudaErrorInvalidValue;
  P.a_load[0] = P.b_load[0] = kLoadK;
  P.tmA[1] = P.tmA[0];
  P.tmB[1] = P.tmB[0];
  P.M[0] = a.chunk;
  P.N[0] = a.V;
  P.K[0] = static_cast<int>(p.d);
  P.bn[0] = kBN;  // the epilogue's 128-column statistic blocks need full 256-wide tiles
  P.tx_bytes[0] = 2u * kStageBytes;
  P.count_mode[0] = 1;
  P.nprob = 1;
  P.n_valid = a.n_valid;
  P.row0 = a.row0;
  P.chunk = a.chunk;
  P.counter = p.counter;
  P.err = p.err;
  P.k2 = p.k2;
  P.V = a.V;
  P.cpad = a.cpad;
  P.n_pb = a.n_pb;
  P.K_top = a.K;
  P.rows = a.rows;
  P.idx_sorted = a.idx_sorted;
  P.p_sorted = a.p_sorted;
  P.boff = a.boff;
  P.part_m = a.part_m;
  P.part_l = a.part_l;
  P.part_ps = a.part_ps;
  P.u = p.u;
  P.ldg = a.ldg;
  if (p.u != nullptr) {  // the stored exponentials leave through the staging buffers
    if (!encode_tmap_store(&P.tmOut[0], p.u, false, a.ldg, a.cpad, a.ldg, 64, 32))
      return cudaErrorInvalidValue;
    P.out_tma[0] = 1;
  }
  if (p.row_ref) {
    if (a.mref == nullptr || a.row_flag == nullptr || p.u == nullptr) return cudaErrorInvalidValue;
    P.mref = a.mref;
    P.row_flag = a.row_flag;
  }
  cudaError_t e = cudaMemsetAsync(p.counter, 0, sizeof(uint32_t), s);
  if (e != cudaSuccess) return e;
  return launch_mode<kModePass1>(P, p.num_sms, s);
}

cudaError_t launch_tc_dual_pass1(const DualPass1Args& p, const ChunkArgs& a, cudaStream_t s) {
  KParams P;
  memset(&P, 0, sizeof(P));
  // problem 0: teacher logits h_t,c W_t^T; problem 1: student logits h_s,c W_s^T
  if (!encode_operand(&P.tmA[0], p.hc_t, kLoadK, p.d_t, a.cpad, p.d_t, kBM) ||
      !encode_operand(&P.tmB[0], p.W_t, kLoadK, p.d_t, a.V, p.d_t, kBN / 2) ||
      !encode_operand(&P.tmA[1], p.hc_s, kLoadK, p.d_s, a.cpad, p.d_s, kBM) ||
      !encode_operand(&P.tmB[1], p.W_s, kLoadK, p.d_s, a.V, p.d_s, kBN / 2))
    return cudaErrorInvalidValue;
  for (int pi = 0; pi < 2; ++pi) {
    P.a_load[pi] = P.b_load[pi] = kLoadK;
    P.M[pi] = a.chunk;
    P.N[pi] = a.V;
    P.bn[pi] = kBN;
    P.tx_bytes[pi] = 2u * kStageBytes;
    P.count_mode[pi] = 1;
  }
  P.K[0] = static_cast<int>(p.d_t);
  P.K[1] = static_cast<int>(p.d_s);
  P.nprob = 2;
  P.n_valid = a.n_valid;
  P.row0 = a.row0;
  P.chunk = a.chunk;
  P.counter = p.counter;
  P.err = p.err;
  P.k2 = p.k2;
  P.V = a.V;
  P.cpad = a.cpad;
  P.n_pb = a.n_pb;
  P.part_m = a.part_m;
  P.part_l = a.part_l;
  P.u = p.u_s;
  P.ldg = a.ldg;
  P.u_t = p.u_t;
  // both exponential tiles leave through the staging buffers: student in
  // tmOut[0], teacher in tmOut[1]
  if (!encode_tmap_store(&P.tmOut[0], p.u_s, false, a.ldg, a.cpad, a.ldg, 64, 32) ||
      !encode_tmap_store(&P.tmOut[1], p.u_t, false, a.ldg, a.cpad, a.ldg, 64, 32))
    return cudaErrorInvalidValue;
  P.part_mt = p.part_mt;
  P.part_lt = p.part_lt;
  P.part_a = p.part_a;
  cudaError_t e = cudaMemsetAsync(p.counter, 0, sizeof(uint32_t), s);
  if (e != cudaSuccess) return e;
  return launch_mode<kModeDual>(P, p.num_sms, s);
}

cudaError_t launch_tc_topk(const TopkGemmArgs& g, int pass, cudaStream_t s) {
  KParams P;
  memset(&P, 0, sizeof(P));
  if (!encode_operand(&P.tmA[0], g.h, kLoadK, g.d, g.count, g.d, kBM) ||
      !encode_operand(&P.tmB[0], g.W, kLoadK, g.d, g.V, g.d, kBN / 2))
    return cudaErrorInvalidValue;
  P.tmA[1] = P.tmA[0];
  P.tmB[1] = P.tmB[0];
  P.a_load[0] = P.b_load[0] = kLoadK;
  P.M[0] = static_cast<int>(g.count);
  P.N[0] = static_cast<int>(g.v_cols);
  P.K[0] = static_cast<int>(g.d);
  P.bn[0] = kBN;  // the epilogue's 128-column blocks need full 256-wide tiles
  P.tx_bytes[0] = 2u * kStageBytes;
  P.nprob = 1;
  P.chunk = static_cast<int>(g.count);
  P.counter = g.counter;
  P.err = g.err;
  P.V = static_cast<int>(g.v_cols);
  P.n_pb = static_cast<int>(ceil_div(g.v_cols, kPB));
  P.bkey = g.bkey;
  P.bkey_ld = ceil_div(g.V, kPB);
  P.gate = g.gate;
  P.tau = g.tau;
  P.cnt = g.cnt;
  P.cand = g.cand;
  P.cap = g.cap;
  cudaError_t e = cudaMemsetAsync(g.counter, 0, sizeof(uint32_t), s);
  if (e != cudaSuccess) return e;
  return pass == 1 ? launch_mode<kModeTopkMax>(P, g.num_sms, s)
                   : launch_mode<kModeTopkCand>(P, g.num_sms, s);
}

}  // namespace kd
