// linear_logp_tc.cu -- tensor-core kernels of linear_logp: the fused forward
// and the two GEMMs of the backward.
//
// Forward ("linear_logp", RL-Kernel issue #101, maintainer comment, P0
// operator list; chain index 7 of PR #264 "docs(ws1): batch-invariance
// contract RFC"):
//   z[t, v] = sum_k h[t, k] W[v, k],  lse[t] = log sum_v exp z[t, v],
//   logp[t] = z[t, target_t] - lse[t];   z never leaves the chip.
// Backward with respect to h (issue #244 "[WS1 Test] ...", Workstream 3 #153:
// fixed, batch-shape-independent reduction order, no atomicAdd):
//   p[t, v]  = exp(z[t, v] - lse[t])
//   dh[t, :] = sum over the row's fp32 entries e of w_e W[v_e, :]
//              - sum_v dZ[t, v] W[v, :]                        (GEMM 2, fp32)
// where the entries are the target column and the columns with p >= 1/64,
// w = g (onehot - p) in fp32, and dZ = g p rounded to bf16 on every other
// column, 0 on those (GEMM 1).  A peaked softmax thus never puts a large,
// bf16-rounded term into the sum.
//
// One persistent, warp-specialised tile kernel serves the three GEMMs.  It
// runs as CTA pairs (clusters of 2 on neighbouring SMs) sharing 256x256 output
// tiles through the pair form of the tensor core (tcgen05 cta_group::2):
//   warp 4      TMA producer (both CTAs): this CTA's 128 rows of A and 128 of
//               the tile's 256 B rows (K-major 128x64, or two MN-major 64x64
//               boxes) per 64-wide K stage, 6-stage ring, 128-byte swizzle;
//               all copies of a stage complete on the even CTA's barrier;
//   warp 5      allocates 512 TMEM columns (both CTAs, collectively); in the
//               even CTA, issues tcgen05.mma (M=256, N=256, K=16, bf16 x bf16
//               -> fp32) into one of two 256-column accumulators, reading A and
//               B from both CTAs' shared memory and writing each CTA's 128
//               rows of D to its own TMEM; commits signal both CTAs;
//   warps 0-3   epilogue (both CTAs): thread i owns row i of its CTA's half
//               (TMEM lane i) and drains one accumulator while the next tile
//               accumulates into the other.
// Epilogues:
//   kFwd  the row's softmax partial over the tile's 256 vocabulary columns,
//         m = max z, s = sum 2^((z - m) log2 e), and z[target] if the target
//         is in the tile, written to workspace[row][tile];
//   kDz   dZ (0 on inactive rows) through TMA stores and, for the fused full
//         backward, dZ^T as well; the row's fp32 entries appended to its list;
//   kDh   dh = (the row's sorted entries) . W - acc in fp32 (0 on inactive rows);
//   kLogits  z rounded to bf16 (the dense path's lm_head);
//   kGreedy  kFwd plus the lowest column holding the tile maximum;
//   kDzT  kDz's output transposed, from z^T = W h^T;
//   kDwK  dW[v, :] = sum over the entries of column v (in canonical token
//         order, fp32) of w h  -  (dZ^T h)[v, :].
// (kDh2 and kDwK2 are kDh and kDwK with two row blocks per tile.)
// A second small kernel (linear_logp_merge) folds the forward partials of a
// row in a fixed order into lse and logp.
//
// Batch invariance by construction: the tile shape, the K order (64-wide
// stages ascending, 16-wide MMAs ascending inside a stage), the epilogue's
// column order and the merge order are identical for every T; a row's results
// depend only on that row's inputs and on W (rows of a tensor-core tile do not
// interact), never on the tile, CTA or M position that holds the row, on the
// schedule, or on how the backward cuts T into chunks.  V is never split
// across CTAs in the backward's sum (no split-K) and no atomics touch results
// (an integer atomicAdd only hands out slots in an entry list, which is then
// sorted by column).
#include <algorithm>
#include <atomic>
#include <cstring>

#include "rk_device.cuh"
#include "rk_internal.h"
#include "token_loss.cuh"

namespace rk {
namespace {

constexpr int BM = 128;  // tile rows per CTA (TMEM lanes); a pair covers 2*BM
constexpr int BN = 256;  // tile columns (TMEM columns per accumulator); each CTA stages BN/2 B rows
constexpr int BK = 64;   // K per pipeline stage (64 bf16 = one 128-byte swizzle row)
constexpr int UK = 16;   // K per tcgen05.mma of kind::f16
constexpr int kStages = 6;
constexpr int kABytes = BM * BK * 2;
constexpr int kBBytes = (BN / 2) * BK * 2;
constexpr uint32_t kTmemCols = 2 * BN;
constexpr int kEpiThreads = 128;
constexpr int kProducerWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kThreads = kEpiThreads + 64;
constexpr int kGroupN = 16;  // raster group (in N tiles) of the forward / dZ GEMMs
constexpr int kGroupNDh = 8;  // raster group (in H tiles) of the dh and dW GEMMs
static_assert(2 * BM == kLiveBlockRows, "a live flag covers one pair tile of rows");

// kFwd: forward partials; kDz: backward GEMM 1; kDh: backward GEMM 2;
// kLogits: the dense path's lm_head (z stored as bf16); kGreedy: kFwd plus
// each tile's argmax column (greedy decoding).
// kDzT: the transpose of kDz's output, dZ^T[v][t] = g[t] exp(z[t, v] - lse[t]),
// from z^T = W h^T (rows = vocabulary, columns = canonical tokens, both
// operands K-major).  kDwK: the weight gradient, dW = S - dZ^T h over
// canonical tokens (A = dZ^T read K-major, B = h read MN-major), S the
// one-hot term added in the epilogue.
// kDh2, kDwK2: kDh and kDwK with two row blocks per tile (see TileCfg).
enum Mode {
    kFwd = 0, kDz = 1, kDh = 2, kLogits = 3, kGreedy = 4, kDzT = 6, kDwK = 7, kDh2 = 8, kDwK2 = 9,
    kFwdS = 10
};
// kFwdS: kFwd that also saves, for the backward, every row's
// e = 2^((z - m_tile) log2 e) in bf16 (the terms of the tile's sum-exp, m_tile
// the row's maximum over the tile) through TMA stores.
__host__ __device__ constexpr bool mode_fwd(int m) { return m == kFwd || m == kFwdS; }
__host__ __device__ constexpr bool mode_dh(int m) { return m == kDh || m == kDh2; }
__host__ __device__ constexpr bool mode_dw(int m) { return m == kDwK || m == kDwK2; }

// Tile queue: the even CTA's producer takes each tile number (from a global
// counter, so that pairs take tiles in the order they become free) and
// publishes it to both CTAs; every other role of the pair reads it there.
constexpr int kTQ = 8;
// readers of a queue slot: the MMA thread and 4 epilogue warps of the even
// CTA, the producer and 4 epilogue warps of the odd CTA
constexpr int kTQReaders = 2 * (kEpiThreads / 32) + 2;

// full / tmem_empty / drain / tq_empty are used in the even CTA only; empty,
// tmem_full and tq_full in both (the MMA commits are multicast to the pair).
struct Ctl {
    uint64_t full[kStages];
    uint64_t empty[kStages];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t drain;
    uint64_t tq_full[kTQ];
    uint64_t tq_empty[kTQ];
    int32_t tq[kTQ];  // tile number, or -1: no more tiles
    uint32_t tmem_base;
    int abort;
};

// kDz with a transposed copy: each epilogue warp stages 32 x 32 bf16 blocks
// (two buffers) for TMA stores of dZ^T.
constexpr int kStageT = 32 * 32;  // elements per staging buffer
constexpr size_t kCtlBytes = (sizeof(Ctl) + 1023) / 1024 * 1024;  // staging stays 1024-aligned
// kDz staging: per epilogue warp two chunk slots of [dZ block, dZ^T block]
constexpr size_t kStageTBytes = (size_t)(kEpiThreads / 32) * 4 * kStageT * 2;

// Per-mode tile shape.  kDh2 and kDwK2 take two row blocks per tile: both
// accumulate into the pair's TMEM at once (columns [0, 256) and [256, 512)),
// so each B stage (the W or h slice, shared across row blocks) is loaded once
// for 2 x 256 rows.  That halves how often the long B stream is read, at the
// cost of the accumulator double buffer; the launchers pick them only for
// long K loops and enough tiles (run_rows).
template <int MODE>
struct TileCfg {
    static constexpr int kMB = (MODE == 8 /* kDh2 */ || MODE == 9 /* kDwK2 */) ? 2 : 1;
    static constexpr int kStg = (kMB == 2) ? 4 : kStages;
    static constexpr int kStgBytes = kMB * kABytes + kBBytes;
    static constexpr size_t kSmem =
        1024 + (size_t)kStg * kStgBytes + kCtlBytes +
        ((MODE == 1 /* kDz */ || MODE == 6 /* kDzT */ || MODE == 10 /* kFwdS */) ? kStageTBytes : 0);
    static_assert(kStg <= kStages, "stage barriers");
    static_assert(kSmem <= 227 * 1024, "shared memory");
};

struct TileArgs {
    // row masking (global row index t = row0 + local row)
    const int64_t *targets;
    const int32_t *cu;
    int32_t num_seqs;
    int64_t row0;
    int64_t rows;  // rows of this launch (local)
    int32_t V;
    int32_t num_m, num_n, num_k;  // num_m counts 256-row pair tiles
    unsigned *err;
    // kFwd
    float2 *part;  // [rows][num_n]
    float *ztgt;   // [rows]
    int32_t *pidx; // kGreedy: [rows][num_n] column of each tile's maximum
    // kDwK (rows = vocabulary, columns = H, K = canonical tokens)
    const int32_t *dw_begin, *dw_end;  // [V] range of each column's entries (empty: no S)
    float *dw;               // [V, H] output, holding S on rows with entries
    int64_t ntok;            // kDzT: number of canonical token positions (columns)
    // tile counter (zeroed before the launch); null: static round-robin order
    unsigned *tile_counter;
    // per 256-row block of the launch: 0 when none of its rows is active, and
    // its tiles are then never handed out (their rows' outputs are written
    // elsewhere); null: every block is computed
    const uint8_t *live;
    // Rounds (non-null; tile_counter is then null): pair p takes tiles p,
    // p + P, p + 2P, ... (P pairs), and starts the tiles of round r only when
    // every pair has issued all copies of round r - 1 (each pair adds one to
    // this counter per round).  The tiles of a round then run in step and
    // share their dZ row blocks and W slices through L2.  Launched
    // cooperatively, so that every pair is resident.
    unsigned *wave_ctr;
    // kDz
    const float *lse;   // [T] (global)
    const float *grad;  // [T] (global)
    uint16_t *dz;       // [rows][ldz] bf16
    int64_t ldz;
    // kDz / kDzT fill, kDh reads: per (local / canonical) row, the entries of
    // the columns kept in fp32 (count, then kEntCap (column, w bits) slots)
    int32_t *ecount;
    int2 *ent;
    // kDh
    const uint16_t *W;  // [V][H]
    float *dh;          // [T][H] (global)
    bool dzT_store;     // kDz: also store dZ^T through the third tensor map
    bool dz_tma;        // kDz / kDzT: store the output through the fourth tensor map
                        // (else plain stores)
    const int64_t *out_rows;  // kDh over canonical rows: physical row of each (or null)
    int32_t H;
};

// Every lane waits; the warp proceeds only if all lanes saw the phase complete,
// so the warp-collective TMEM loads that follow are never reached divergently.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          unsigned *err) {
    const bool ok = mbar_wait(bar, parity, abort, err);
    return __all_sync(0xffffffffu, ok) != 0;
}

// The backward's fp32 terms.  The target column and columns with
// p >= kEntTau (in_fp32) leave the bf16 matrix (0 there) and go to the row's
// entry list as (column, g (onehot - p)).  A list that would overflow can only
// come from an lse that does not belong to the inputs: the term is then
// dropped and RK_DEVERR_LSE raised.
__device__ __forceinline__ bool in_fp32(float p, int64_t col, int64_t tgt, int64_t V) {
    return col < V && (col == tgt || p >= kEntTau);
}

__device__ __noinline__ void emit_entry(float g, float p, int64_t col, int64_t tgt,
                                        int32_t *count, int2 *list, unsigned *err) {
    const float w = __fmul_rn(g, __fsub_rn(col == tgt ? 1.f : 0.f, p));
    const int slot = atomicAdd(count, 1);
    if (slot < kEntCap)
        list[slot] = make_int2((int)col, __float_as_int(w));
    else
        atomicOr(err, kErrLse);
}

template <int MODE>
__device__ __forceinline__ void tile_coords(int64_t tile, const TileArgs &a, int &mb, int &nb) {
    if constexpr (mode_dh(MODE) || mode_dw(MODE)) {
        // groups of kGroupNDh H tiles; inside a group, row blocks outer: CTAs
        // running together share A (dZ rows) and walk W's K (vocabulary) rows
        // in step.  mb counts tiles of TileCfg::kMB row blocks.
        const int64_t nm = (a.num_m + TileCfg<MODE>::kMB - 1) / TileCfg<MODE>::kMB;
        const int64_t per_group = nm * kGroupNDh;
        const int64_t g = tile / per_group;
        const int64_t r = tile - g * per_group;
        const int n0 = (int)g * kGroupNDh;
        const int gn = min(kGroupNDh, a.num_n - n0);
        mb = (int)(r / gn);
        nb = n0 + (int)(r % gn);
    } else {
        const int64_t per_group = (int64_t)a.num_m * kGroupN;
        const int64_t g = tile / per_group;
        const int64_t r = tile - g * per_group;
        const int n0 = (int)g * kGroupN;
        const int gn = min(kGroupN, a.num_n - n0);
        mb = (int)(r / gn);
        nb = n0 + (int)(r % gn);
    }
}

// Rounds of tiles (TileArgs::wave_ctr).  Before tile t (round t / npairs),
// the pair signals every round up to that one and waits until all npairs
// pairs have signalled it; a pair with no more tiles (t >= total) signals all
// remaining rounds and returns.  Bounded: after kWaitLimitNs the pair raises
// the abort flag and RK_DEVERR_TIMEOUT, signals the remaining rounds (so the
// others are not held) and returns false.
__device__ __noinline__ bool wait_round(unsigned *ctr, int64_t t, int64_t total, int64_t npairs,
                                        int64_t &arrived, volatile int *abort, unsigned *err) {
    const int64_t rounds = (total + npairs - 1) / npairs;
    const int64_t rnd = t < total ? t / npairs : rounds - 1;
    for (; arrived < rnd; ++arrived) atomicAdd(ctr, 1u);
    if (t >= total) return true;
    const unsigned need = (unsigned)(npairs * rnd);
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 0; *reinterpret_cast<volatile unsigned *>(ctr) < need; ++i) {
        if ((i & 63u) == 0 && (*abort || global_timer_ns() - t0 > kWaitLimitNs)) {
            *abort = 1;
            atomicOr(err, kErrTimeout);
            for (; arrived < rounds - 1; ++arrived) atomicAdd(ctr, 1u);
            return false;
        }
    }
    return true;
}

// Whether a tile holds an active row (any of its TileCfg::kMB row blocks).
template <int MODE>
__device__ __forceinline__ bool tile_live(int64_t tile, const TileArgs &a) {
    if (a.live == nullptr) return true;
    int mb, nb;
    tile_coords<MODE>(tile, a, mb, nb);
#pragma unroll
    for (int j = 0; j < TileCfg<MODE>::kMB; ++j) {
        const int64_t b = (int64_t)mb * TileCfg<MODE>::kMB + j;
        if (b < a.num_m && a.live[b] != 0) return true;
    }
    return false;
}

template <int MODE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    linear_logp_tiles(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmD,
                      const TileArgs a) {
    // kDh: B is W read as [K = vocabulary rows, N = H columns] (N contiguous,
    // "MN-major"), staged as two 64-column boxes of BK rows per CTA.
    constexpr bool kBmn = mode_dh(MODE) || mode_dw(MODE);
    constexpr uint32_t kIdesc = idesc_bf16_f32(2 * BM, BN, false, kBmn);
    constexpr uint32_t kBBoxBytes = BK * 64 * 2;  // one 64-column MN-major box
    // Descriptor strides.  K-major, 128B swizzle: 8-row groups 1024 B apart;
    // the next 16-wide K slice starts 32 B further.  MN-major, 128B swizzle:
    // 64-column atoms kBBoxBytes apart (leading offset), 8-row K groups 1024 B
    // apart (stride offset); the next 16-row K slice starts 16*128 B further.
    constexpr uint32_t kBLbo = kBmn ? kBBoxBytes : 16;
    constexpr uint32_t kBStepK = kBmn ? (UK * 128) : (UK * 2);
    constexpr uint32_t kALbo = 16;        // A is always K-major
    constexpr uint32_t kAStepK = UK * 2;
    constexpr int kMB = TileCfg<MODE>::kMB;
    constexpr int kStg = TileCfg<MODE>::kStg;
    constexpr int kStgBytes = TileCfg<MODE>::kStgBytes;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    Ctl *ctl = reinterpret_cast<Ctl *>(smem + (size_t)kStg * kStgBytes);
    uint16_t *stageT = reinterpret_cast<uint16_t *>(smem + (size_t)kStg * kStgBytes + kCtlBytes);
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0: issues the MMAs
    const int64_t pair = blockIdx.x >> 1;
    const int64_t npairs = gridDim.x >> 1;
    const int64_t total = (int64_t)((a.num_m + kMB - 1) / kMB) * a.num_n;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&ctl->full[s]), 1);
            mbar_init(smem_u32(&ctl->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&ctl->tmem_full[b]), 1);
            mbar_init(smem_u32(&ctl->tmem_empty[b]), 2 * (kEpiThreads / 32));
        }
        mbar_init(smem_u32(&ctl->drain), 1);
        for (int i = 0; i < kTQ; ++i) {
            mbar_init(smem_u32(&ctl->tq_full[i]), 1);
            mbar_init(smem_u32(&ctl->tq_empty[i]), kTQReaders);
        }
        ctl->abort = 0;
        fence_mbar_init();
    }
    if (warp == kProducerWarp && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == kMmaWarp) {
        tmem_alloc_pair(smem_u32(&ctl->tmem_base), kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers initialised, TMEM allocated
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    volatile int *abort = &ctl->abort;

    if (warp == kProducerWarp) {
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            uint32_t last_ph[kStages];
            bool used[kStages];
            for (int i = 0; i < kStages; ++i) {
                used[i] = false;
                last_ph[i] = 0;
            }
            bool ok = true;
            int q = 0;
            uint32_t qph = 0;
            int64_t next_static = pair;
            int64_t rounds_arrived = 0;  // wave_ctr: rounds this pair has signalled
            while (ok) {
                int32_t tv;
                if (rank == 0) {
                    // take the next tile and publish it to both CTAs
                    if (!mbar_wait_cluster(smem_u32(&ctl->tq_empty[q]), qph ^ 1u, abort, a.err)) {
                        ok = false;
                        break;
                    }
                    // the next tile that holds an active row
                    int64_t t;
                    for (;;) {
                        if (a.tile_counter) {
                            t = (int64_t)atomicAdd(a.tile_counter, 1u);
                        } else {
                            t = next_static;
                            next_static += npairs;
                        }
                        if (t >= total || tile_live<MODE>(t, a)) break;
                    }
                    if (a.wave_ctr != nullptr && !wait_round(a.wave_ctr, t, total, npairs,
                                                             rounds_arrived, abort, a.err))
                        t = total;  // gave up: no more tiles for this pair
                    tv = t < total ? (int32_t)t : -1;
                    for (uint32_t r = 0; r < 2; ++r) {
                        st_shared_cluster_u32(mapa_shared(smem_u32(&ctl->tq[q]), r), (uint32_t)tv);
                        mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->tq_full[q]), r));
                    }
                } else {
                    if (!mbar_wait_cluster(smem_u32(&ctl->tq_full[q]), qph, abort, a.err)) {
                        ok = false;
                        break;
                    }
                    tv = ctl->tq[q];
                    mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->tq_empty[q]), 0));
                }
                if (++q == kTQ) {
                    q = 0;
                    qph ^= 1u;
                }
                if (tv < 0) break;
                const int64_t tile = tv;
                int mb, nb;
                tile_coords<MODE>(tile, a, mb, nb);
                const int arow = mb * kMB * 2 * BM + (int)rank * BM;  // this CTA's A rows
                const int bn0 = nb * BN + (int)rank * (BN / 2);    // this CTA's B rows / H columns
                int nbox0 = 0, nbox1 = 0;    // B boxes of CTA 0 / 1 (MN-major)
                if constexpr (kBmn) {
                    nbox0 = max(0, min(2, (a.H - nb * BN) / 64));
                    nbox1 = max(0, min(2, (a.H - nb * BN - BN / 2) / 64));
                }
                for (int kb = 0; kb < a.num_k; ++kb) {
                    if (!mbar_wait(smem_u32(&ctl->empty[s]), ph ^ 1u, abort, a.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = mapa_shared(smem_u32(&ctl->full[s]), 0);
                    const uint32_t sa = sbase + (uint32_t)(s * kStgBytes);
                    if (rank == 0) {
                        uint32_t bytes = (uint32_t)(2 * kStgBytes);
                        if constexpr (kBmn)
                            bytes = (uint32_t)(2 * kMB * kABytes + (nbox0 + nbox1) * (int)kBBoxBytes);
                        mbar_arrive_expect_tx(smem_u32(&ctl->full[s]), bytes);
                    }
                    if constexpr (kBmn) {
#pragma unroll
                        for (int j = 0; j < kMB; ++j)
                            tma_load_2d_pair(sa + j * kABytes, &tmA, fb, kb * BK, arow + j * 2 * BM);
                        const int nbox = rank == 0 ? nbox0 : nbox1;
                        for (int j = 0; j < nbox; ++j)
                            tma_load_2d_pair(sa + kMB * kABytes + j * kBBoxBytes, &tmB, fb,
                                             bn0 + j * 64, kb * BK);
                    } else {
                        tma_load_2d_pair(sa, &tmA, fb, kb * BK, arow);
                        tma_load_2d_pair(sa + kABytes, &tmB, fb, kb * BK, bn0);
                    }
                    used[s] = true;
                    last_ph[s] = ph;
                    if (++s == kStg) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (rank == 0 && a.wave_ctr != nullptr) {
                // every round signalled, however the loop ended, so that no
                // other pair waits for this one
                const int64_t rounds = (total + npairs - 1) / npairs;
                for (; rounds_arrived < rounds - 1; ++rounds_arrived) atomicAdd(a.wave_ctr, 1u);
            }
            if (!ok) {  // let every issued copy land before the pair exits
                if (rank == 0) {
                    for (int i = 0; i < kStages; ++i)
                        if (used[i])
                            mbar_wait_drain(smem_u32(&ctl->full[i]), last_ph[i], 100000000ull);
                } else {
                    const uint64_t t0 = global_timer_ns();
                    while (global_timer_ns() - t0 < 2000000ull) {
                    }
                }
            }
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0 && rank == 0) {
            int s = 0;
            uint32_t ph = 0;
            int b = 0;
            uint32_t tph = 0;
            bool ok = true;
            int q = 0;
            uint32_t qph = 0;
            while (ok) {
                if (!mbar_wait_cluster(smem_u32(&ctl->tq_full[q]), qph, abort, a.err)) break;
                const int32_t tv = ctl->tq[q];
                mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->tq_empty[q]), 0));
                if (++q == kTQ) {
                    q = 0;
                    qph ^= 1u;
                }
                if (tv < 0) break;
                if (!mbar_wait(smem_u32(&ctl->tmem_empty[b]), tph ^ 1u, abort, a.err)) break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(b * BN);
                for (int kb = 0; kb < a.num_k; ++kb) {
                    if (!mbar_wait(smem_u32(&ctl->full[s]), ph, abort, a.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = sbase + (uint32_t)(s * kStgBytes);
                    const uint64_t bd = smem_desc_sw128(sa + kMB * kABytes, kBLbo, 1024);
#pragma unroll
                    for (int kk = 0; kk < BK / UK; ++kk) {
#pragma unroll
                        for (int j = 0; j < kMB; ++j) {
                            const uint64_t ad = smem_desc_sw128(sa + j * kABytes, kALbo, 1024);
                            mma_bf16_ss_pair(d + (uint32_t)(j * BN), ad + (uint64_t)((kk * kAStepK) >> 4),
                                             bd + (uint64_t)((kk * kBStepK) >> 4), kIdesc,
                                             (kb | kk) != 0 ? 1u : 0u);
                        }
                    }
                    mma_commit_pair(smem_u32(&ctl->empty[s]), 0x3);
                    if (++s == kStg) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit_pair(smem_u32(&ctl->tmem_full[b]), 0x3);
                // two accumulator buffers, or one holding kMB = 2 row blocks
                if (++b == 2 / kMB) {
                    b = 0;
                    tph ^= 1u;
                }
            }
            // No MMA may still be reading shared memory or writing TMEM when
            // the pair releases them.
            mma_commit_pair(smem_u32(&ctl->drain), 0x1);
            mbar_wait_drain(smem_u32(&ctl->drain), 0, 1000000000ull);
        }
    } else {
        // Epilogue: warp w reads TMEM lanes [32w, 32w+32) = rows of this CTA's half.
        int b = 0;
        uint32_t tph = 0;
        uint32_t tchunks = 0;  // transposed blocks stored by this warp so far
        const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
        int q = 0;
        uint32_t qph = 0;
        for (;;) {
            // every lane waits, as in warp_wait
            const bool got = mbar_wait_cluster(smem_u32(&ctl->tq_full[q]), qph, abort, a.err);
            if (__all_sync(0xffffffffu, got) == 0) break;
            const int32_t tv = ctl->tq[q];
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&ctl->tq_empty[q]), 0));
            if (++q == kTQ) {
                q = 0;
                qph ^= 1u;
            }
            if (tv < 0) break;
            const int64_t tile = tv;
            int mb, nb;
            tile_coords<MODE>(tile, a, mb, nb);
            const int64_t lrow = (int64_t)mb * 2 * BM + (int64_t)rank * BM + threadIdx.x;  // local row
            const bool in_range = lrow < a.rows;
            const int64_t grow = a.row0 + lrow;                    // global row
            // the row's target (forward and dZ tiles only: kDzT rows are vocabulary rows)
            const int64_t tgt = ((mode_fwd(MODE) || MODE == kDz) && in_range && a.targets != nullptr)
                                    ? a.targets[grow]
                                    : -1;
            const int n0 = nb * BN;
            const uint32_t empty_bar = mapa_shared(smem_u32(&ctl->tmem_empty[b]), 0);
            if constexpr (mode_fwd(MODE) || MODE == kGreedy) {
                const int valid = min(BN, a.V - n0);
                const int tcol = (tgt >= n0 && tgt < (int64_t)n0 + valid) ? (int)(tgt - n0) : -1;
                if (!warp_wait(smem_u32(&ctl->tmem_full[b]), tph, abort, a.err)) break;
                tc_fence_after();
                const uint32_t taddr = tmem + lane_off + (uint32_t)(b * BN);
                // pass 1: the row's maximum over the tile (and, greedy, its
                // lowest column: a later column replaces it only if strictly larger)
                float m = -INFINITY;
                int arg = 0;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr + (uint32_t)(c * 32), r);
                    tmem_ld_wait();
                    if constexpr (MODE == kGreedy) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const float x = __uint_as_float(r[j]);
                            if (c * 32 + j < valid && x > m) {
                                m = x;
                                arg = c * 32 + j;
                            }
                        }
                    } else if (valid == BN) {
#pragma unroll
                        for (int j = 0; j < 32; ++j) m = fmaxf(m, __uint_as_float(r[j]));
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (c * 32 + j < valid) m = fmaxf(m, __uint_as_float(r[j]));
                    }
                }
                // pass 2: sum of 2^((z - m) log2 e), four accumulators in a fixed pattern
                const float mb2 = __fmul_rn(-m, kLog2e);
                float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
                float zt = 0.f;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr + (uint32_t)(c * 32), r);
                    tmem_ld_wait();
                    float e[32];
                    if (valid == BN) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            e[j] = ex2(__fmaf_rn(__uint_as_float(r[j]), kLog2e, mb2));
                    } else {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            e[j] = (c * 32 + j < valid)
                                       ? ex2(__fmaf_rn(__uint_as_float(r[j]), kLog2e, mb2))
                                       : 0.f;
                    }
#pragma unroll
                    for (int j = 0; j < 32; j += 4) {
                        acc0 = __fadd_rn(acc0, e[j]);
                        acc1 = __fadd_rn(acc1, e[j + 1]);
                        acc2 = __fadd_rn(acc2, e[j + 2]);
                        acc3 = __fadd_rn(acc3, e[j + 3]);
                    }
                    if constexpr (MODE == kFwdS) {
                        // the warp's 32 x 32 block of e, in bf16, through one TMA
                        // store (clipped at V and at the rows), staged as in kDz
                        uint16_t *sbz = stageT + (warp * 4 + (int)(tchunks & 1) * 2) * kStageT;
                        if (lane == 0 && tchunks >= 2) bulk_wait_group_read<1>();
                        __syncwarp();
                        uint8_t *rowp = reinterpret_cast<uint8_t *>(sbz) + lane * 64;
                        const int sw = (lane >> 1) & 3;
#pragma unroll
                        for (int qq = 0; qq < 4; ++qq)
                            *reinterpret_cast<uint4 *>(rowp + ((qq ^ sw) << 4)) = make_uint4(
                                pack_bf16x2(e[8 * qq], e[8 * qq + 1]), pack_bf16x2(e[8 * qq + 2], e[8 * qq + 3]),
                                pack_bf16x2(e[8 * qq + 4], e[8 * qq + 5]), pack_bf16x2(e[8 * qq + 6], e[8 * qq + 7]));
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            const int64_t r0 = (int64_t)mb * 2 * BM + (int64_t)rank * BM + warp * 32;
                            tma_store_2d(&tmD, smem_u32(sbz), n0 + c * 32, (int32_t)r0);
                            bulk_commit_group();
                        }
                        ++tchunks;
                    }
                    const int rel = tcol - c * 32;
                    if (rel >= 0 && rel < 32) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            if (j == rel) zt = __uint_as_float(r[j]);
                    }
                }
                const float s = __fadd_rn(__fadd_rn(acc0, acc1), __fadd_rn(acc2, acc3));
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(empty_bar);
                if (in_range) {
                    a.part[lrow * a.num_n + nb] = make_float2(m, s);
                    if (tcol >= 0) a.ztgt[lrow] = zt;
                    if constexpr (MODE == kGreedy) a.pidx[lrow * a.num_n + nb] = n0 + arg;
                }
            } else if constexpr (MODE == kDz || MODE == kLogits) {
                constexpr bool kSoft = (MODE == kDz);
                const bool active =
                    in_range && (!kSoft || row_active(grow, tgt, a.cu, a.num_seqs));
                const float g = (kSoft && active) ? a.grad[grow] : 0.f;
                const float nl = (kSoft && active) ? __fmul_rn(-a.lse[grow], kLog2e) : 0.f;
                const int valid = min(BN, a.V - n0);
                // the target's column within this tile (or out of [0, BN))
                const int trel = (tgt >= n0 && tgt < (int64_t)n0 + BN) ? (int)(tgt - n0) : -1;
                if (!warp_wait(smem_u32(&ctl->tmem_full[b]), tph, abort, a.err)) break;
                tc_fence_after();
                const uint32_t taddr = tmem + lane_off + (uint32_t)(b * BN);
                uint16_t *drow = a.dz + lrow * a.ldz + n0;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr + (uint32_t)(c * 32), r);
                    tmem_ld_wait();
                    uint32_t pk[16];
                    uint32_t big = 0;  // kDz: columns of this chunk kept in fp32
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        float d0, d1;
                        if constexpr (kSoft) {
                            const float p0 = ex2(__fmaf_rn(__uint_as_float(r[2 * j]), kLog2e, nl));
                            const float p1 =
                                ex2(__fmaf_rn(__uint_as_float(r[2 * j + 1]), kLog2e, nl));
                            // 32-bit test of in_fp32 relative to the tile
                            const int k0 = c * 32 + 2 * j;
                            const bool b0 = active && k0 < valid && (k0 == trel || p0 >= kEntTau);
                            const bool b1 =
                                active && k0 + 1 < valid && (k0 + 1 == trel || p1 >= kEntTau);
                            big |= (b0 ? 1u : 0u) << (2 * j);
                            big |= (b1 ? 1u : 0u) << (2 * j + 1);
                            d0 = (active && !b0) ? __fmul_rn(g, p0) : 0.f;
                            d1 = (active && !b1) ? __fmul_rn(g, p1) : 0.f;
                        } else {
                            d0 = __uint_as_float(r[2 * j]);
                            d1 = __uint_as_float(r[2 * j + 1]);
                        }
                        pk[j] = pack_bf16x2(d0, d1);
                    }
                    if constexpr (kSoft) {
                        if (big) {  // rare: the target's tile, or a large p
#pragma unroll
                            for (int k = 0; k < 32; ++k)
                                if ((big >> k) & 1u)
                                    emit_entry(g, ex2(__fmaf_rn(__uint_as_float(r[k]), kLog2e, nl)),
                                               (int64_t)n0 + c * 32 + k, tgt, a.ecount + lrow,
                                               a.ent + lrow * kEntCap, a.err);
                        }
                    }
                    if constexpr (kSoft) {
                        if (a.dz_tma || a.dzT_store) {
                            // The warp's 32 x 32 block goes out through TMA
                            // stores (clipped at V and at the row count): dZ
                            // from rows of 64 bytes with the 64-byte swizzle
                            // (16-byte chunk q of row r at chunk q ^ ((r >> 1) & 3),
                            // so a quarter-warp's writes hit distinct banks),
                            // and dZ^T[n0 + c*32 + j][token] transposed.
                            uint16_t *sbz = stageT + (warp * 4 + (int)(tchunks & 1) * 2) * kStageT;
                            uint16_t *sbt = sbz + kStageT;
                            if (lane == 0 && tchunks >= 2) bulk_wait_group_read<1>();
                            __syncwarp();
                            if (a.dz_tma) {
                                uint8_t *rowp = reinterpret_cast<uint8_t *>(sbz) + lane * 64;
                                const int sw = (lane >> 1) & 3;
#pragma unroll
                                for (int qq = 0; qq < 4; ++qq)
                                    *reinterpret_cast<uint4 *>(rowp + ((qq ^ sw) << 4)) =
                                        make_uint4(pk[4 * qq], pk[4 * qq + 1], pk[4 * qq + 2], pk[4 * qq + 3]);
                            }
                            if (a.dzT_store) {
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    sbt[j * 32 + lane] =
                                        (uint16_t)((j & 1) ? (pk[j >> 1] >> 16) : (pk[j >> 1] & 0xFFFFu));
                            }
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                const int64_t tok0 = (int64_t)mb * 2 * BM + (int64_t)rank * BM + warp * 32;
                                if (a.dz_tma) tma_store_2d(&tmD, smem_u32(sbz), n0 + c * 32, (int32_t)tok0);
                                if (a.dzT_store) tma_store_2d(&tmC, smem_u32(sbt), (int32_t)tok0, n0 + c * 32);
                                bulk_commit_group();
                            }
                            ++tchunks;
                        }
                    }
                    if (in_range && !(kSoft && a.dz_tma)) {
                        const int c0 = c * 32;
                        if (c0 + 32 <= valid) {
                            uint4 *dst = reinterpret_cast<uint4 *>(drow + c0);
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                if (c0 + j < valid)
                                    drow[c0 + j] = (uint16_t)((j & 1) ? (pk[j >> 1] >> 16) : (pk[j >> 1] & 0xFFFFu));
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(empty_bar);
            } else if constexpr (MODE == kDzT) {
                // rows = vocabulary v, columns = canonical tokens; each column
                // brings its own lse and g (tokens past the active count have g = 0)
                const bool vrow = lrow < a.V;
                const int tvalid = (int)(a.ntok - n0 < (int64_t)BN ? a.ntok - n0 : (int64_t)BN);
                if (!warp_wait(smem_u32(&ctl->tmem_full[b]), tph, abort, a.err)) break;
                tc_fence_after();
                const uint32_t taddr = tmem + lane_off + (uint32_t)(b * BN);
                uint16_t *drow = a.dz + lrow * a.ldz + n0;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t r[32];
                    tmem_ld_32x32b_x32(taddr + (uint32_t)(c * 32), r);
                    tmem_ld_wait();
                    const int c0 = c * 32;
                    if (c0 < tvalid) {  // the same for the whole warp
                        // lane j holds token column c0 + j's target, -lse log2e and g
                        const bool okl = c0 + lane < tvalid;
                        const int tl = n0 + c0 + lane;
                        const int tgl = okl ? (int)a.targets[tl] : -1;
                        const float nll = okl ? __fmul_rn(-a.lse[tl], kLog2e) : 0.f;
                        const float gl = okl ? a.grad[tl] : 0.f;
                        uint32_t pk[16];
                        uint32_t big = 0;
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            const int tg0 = __shfl_sync(0xffffffffu, tgl, 2 * j);
                            const int tg1 = __shfl_sync(0xffffffffu, tgl, 2 * j + 1);
                            const float nl0 = __shfl_sync(0xffffffffu, nll, 2 * j);
                            const float nl1 = __shfl_sync(0xffffffffu, nll, 2 * j + 1);
                            const float g0 = __shfl_sync(0xffffffffu, gl, 2 * j);
                            const float g1 = __shfl_sync(0xffffffffu, gl, 2 * j + 1);
                            const float p0 = ex2(__fmaf_rn(__uint_as_float(r[2 * j]), kLog2e, nl0));
                            const float p1 = ex2(__fmaf_rn(__uint_as_float(r[2 * j + 1]), kLog2e, nl1));
                            // token t's fp32 entries, as kDz makes them for row t
                            const bool a0 = vrow && tg0 >= 0, a1 = vrow && tg1 >= 0;
                            const bool b0 = a0 && in_fp32(p0, lrow, tg0, a.V);
                            const bool b1 = a1 && in_fp32(p1, lrow, tg1, a.V);
                            big |= (b0 ? 1u : 0u) << (2 * j);
                            big |= (b1 ? 1u : 0u) << (2 * j + 1);
                            pk[j] = pack_bf16x2((a0 && !b0) ? __fmul_rn(g0, p0) : 0.f,
                                                (a1 && !b1) ? __fmul_rn(g1, p1) : 0.f);
                        }
                        if (__any_sync(0xffffffffu, big != 0)) {  // rare
#pragma unroll
                            for (int k = 0; k < 32; ++k) {
                                const int tgk = __shfl_sync(0xffffffffu, tgl, k);
                                const float nlk = __shfl_sync(0xffffffffu, nll, k);
                                const float gk = __shfl_sync(0xffffffffu, gl, k);
                                if ((big >> k) & 1u) {
                                    const int tk = n0 + c0 + k;
                                    emit_entry(gk, ex2(__fmaf_rn(__uint_as_float(r[k]), kLog2e, nlk)),
                                               lrow, tgk, a.ecount + tk, a.ent + (int64_t)tk * kEntCap,
                                               a.err);
                                }
                            }
                        }
                        if (a.dz_tma) {
                            // the warp's 32 x 32 block through one TMA store, as
                            // in kDz (rows past V and tokens past ntok are clipped)
                            uint16_t *sbz = stageT + (warp * 4 + (int)(tchunks & 1) * 2) * kStageT;
                            if (lane == 0 && tchunks >= 2) bulk_wait_group_read<1>();
                            __syncwarp();
                            uint8_t *rowp = reinterpret_cast<uint8_t *>(sbz) + lane * 64;
                            const int sw = (lane >> 1) & 3;
#pragma unroll
                            for (int qq = 0; qq < 4; ++qq)
                                *reinterpret_cast<uint4 *>(rowp + ((qq ^ sw) << 4)) =
                                    make_uint4(pk[4 * qq], pk[4 * qq + 1], pk[4 * qq + 2], pk[4 * qq + 3]);
                            fence_proxy_async_smem();
                            __syncwarp();
                            if (lane == 0) {
                                const int64_t v0 = (int64_t)mb * 2 * BM + (int64_t)rank * BM + warp * 32;
                                tma_store_2d(&tmD, smem_u32(sbz), n0 + c0, (int32_t)v0);
                                bulk_commit_group();
                            }
                            ++tchunks;
                        } else if (vrow) {
                            if (c0 + 32 <= tvalid) {
                                uint4 *dst = reinterpret_cast<uint4 *>(drow + c0);
#pragma unroll
                                for (int q = 0; q < 4; ++q)
                                    dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
                            } else {
#pragma unroll
                                for (int j = 0; j < 32; ++j)
                                    if (c0 + j < tvalid)
                                        drow[c0 + j] = (uint16_t)((j & 1) ? (pk[j >> 1] >> 16) : (pk[j >> 1] & 0xFFFFu));
                            }
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(empty_bar);
            } else if constexpr (mode_dw(MODE)) {
                if (!warp_wait(smem_u32(&ctl->tmem_full[b]), tph, abort, a.err)) break;
                tc_fence_after();
#pragma unroll 1
                for (int j = 0; j < kMB; ++j) {
                    // vrow is a vocabulary row; its fp32 term S (the entries of
                    // column vr: the tokens whose target it is or where its
                    // p >= kEntTau, in canonical token order) is already in dW
                    const int64_t vr = ((int64_t)mb * kMB + j) * 2 * BM + (int64_t)rank * BM + threadIdx.x;
                    const bool vrow = vr < a.V;
                    const int32_t b0 = vrow ? a.dw_begin[vr] : 0;
                    const int32_t b1 = vrow ? a.dw_end[vr] : 0;
                    const int hvalid = min(BN, a.H - n0);
                    const uint32_t taddr = tmem + lane_off + (uint32_t)((b + j) * BN);
                    float *orow = a.dw + vr * (int64_t)a.H + n0;
#pragma unroll 1
                    for (int c = 0; c < BN / 32; ++c) {
                        uint32_t r[32];
                        tmem_ld_32x32b_x32(taddr + (uint32_t)(c * 32), r);
                        tmem_ld_wait();
                        if (vrow && c * 32 < hvalid) {
                            // the fp32 term S, already in dW for rows with entries
                            float sacc[32];
                            if (b1 > b0) {
                                const float4 *src = reinterpret_cast<const float4 *>(orow + c * 32);
#pragma unroll
                                for (int qq = 0; qq < 8; ++qq) {
                                    const float4 v4 = src[qq];
                                    sacc[4 * qq] = v4.x;
                                    sacc[4 * qq + 1] = v4.y;
                                    sacc[4 * qq + 2] = v4.z;
                                    sacc[4 * qq + 3] = v4.w;
                                }
                            } else {
#pragma unroll
                                for (int jj = 0; jj < 32; ++jj) sacc[jj] = 0.f;
                            }
                            float4 *dst = reinterpret_cast<float4 *>(orow + c * 32);
#pragma unroll
                            for (int qq = 0; qq < 8; ++qq)
                                dst[qq] = make_float4(
                                    __fsub_rn(sacc[4 * qq], __uint_as_float(r[4 * qq])),
                                    __fsub_rn(sacc[4 * qq + 1], __uint_as_float(r[4 * qq + 1])),
                                    __fsub_rn(sacc[4 * qq + 2], __uint_as_float(r[4 * qq + 2])),
                                    __fsub_rn(sacc[4 * qq + 3], __uint_as_float(r[4 * qq + 3])));
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(empty_bar);
            } else {  // kDh, kDh2
                if (!warp_wait(smem_u32(&ctl->tmem_full[b]), tph, abort, a.err)) break;
                tc_fence_after();
#pragma unroll 1
                for (int j = 0; j < kMB; ++j) {
                    const int64_t lr = ((int64_t)mb * kMB + j) * 2 * BM + (int64_t)rank * BM + threadIdx.x;
                    const bool inr = lr < a.rows;
                    const int64_t gr = a.row0 + lr;
                    const int64_t tg = inr ? a.targets[gr] : -1;
                    const bool active = inr && row_active(gr, tg, a.cu, a.num_seqs) && tg < a.V;
                    // the row's fp32 entries (target column, columns with
                    // p >= kEntTau), sorted by column
                    const int cnt = active ? min(a.ecount[lr], kEntCap) : 0;
                    const int2 *el = a.ent + lr * kEntCap;
                    const int2 e0 = cnt > 0 ? el[0] : make_int2(0, 0);  // usually the only one
                    const int hvalid = min(BN, a.H - n0);  // a multiple of 64
                    // canonical rows scatter to their physical rows; padding
                    // positions (inactive) are not stored
                    const bool store = inr && (a.out_rows == nullptr || active);
                    const int64_t orow_i = (a.out_rows == nullptr) ? gr : (active ? a.out_rows[gr] : 0);
                    const uint32_t taddr = tmem + lane_off + (uint32_t)((b + j) * BN);
                    float *orow = a.dh + orow_i * (int64_t)a.H + n0;
#pragma unroll 1
                    for (int c = 0; c < BN / 32; ++c) {
                        uint32_t r[32];
                        tmem_ld_32x32b_x32(taddr + (uint32_t)(c * 32), r);
                        tmem_ld_wait();
                        if (store && c * 32 < hvalid) {
                            float o[32];
                            if (active) {
                                float sacc[32];
#pragma unroll
                                for (int jj = 0; jj < 32; ++jj) sacc[jj] = 0.f;
                                for (int e = 0; e < cnt; ++e) {
                                    const int2 en = (e == 0) ? e0 : el[e];
                                    const float w = __int_as_float(en.y);
                                    const uint4 *src = reinterpret_cast<const uint4 *>(
                                        a.W + (int64_t)en.x * a.H + n0 + c * 32);
#pragma unroll
                                    for (int qq = 0; qq < 4; ++qq) {
                                        const uint4 v4 = __ldg(src + qq);
                                        const uint32_t w4[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
                                        for (int u = 0; u < 4; ++u) {
                                            const int jj = qq * 8 + u * 2;
                                            sacc[jj] = __fmaf_rn(w, bf16_lo(w4[u]), sacc[jj]);
                                            sacc[jj + 1] = __fmaf_rn(w, bf16_hi(w4[u]), sacc[jj + 1]);
                                        }
                                    }
                                }
#pragma unroll
                                for (int jj = 0; jj < 32; ++jj) o[jj] = __fsub_rn(sacc[jj], __uint_as_float(r[jj]));
                            } else {
#pragma unroll
                                for (int jj = 0; jj < 32; ++jj) o[jj] = 0.f;
                            }
                            float4 *dst = reinterpret_cast<float4 *>(orow + c * 32);
#pragma unroll
                            for (int qq = 0; qq < 8; ++qq)
                                dst[qq] = make_float4(o[4 * qq], o[4 * qq + 1], o[4 * qq + 2], o[4 * qq + 3]);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(empty_bar);
            }
            if (++b == 2 / kMB) {
                b = 0;
                tph ^= 1u;
            }
        }
    }

    if constexpr (MODE == kDz || MODE == kDzT || MODE == kFwdS) {
        // staged blocks must be read out of shared memory and written
        if (warp < kEpiThreads / 32 && lane == 0 && (a.dzT_store || a.dz_tma || MODE == kFwdS))
            bulk_wait_group_all();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the pair is done with its shared memory and TMEM
    if (warp == kMmaWarp) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc_pair(tmem, kTmemCols);
    }
}

constexpr int kMergeRowsPerBlock = 8;

// The row's log-sum-exp from its tile partials: lane l folds tiles l, l+32,
// ... in ascending order, then a fixed xor tree; every lane ends with the
// same (m, s).  Shared by the forward and greedy merges, so a greedy step and
// a later scoring of its token give the same lse bit for bit.
__device__ __forceinline__ void fold_tiles(const float2 *__restrict__ pr, int num_n, int lane,
                                           float &m, float &s) {
    m = -INFINITY;
    s = 0.f;
#pragma unroll 4
    for (int j = lane; j < num_n; j += 32) {
        const float2 p = pr[j];
        lse_merge(m, s, p.x, p.y);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, m, off);
        const float so = __shfl_xor_sync(0xffffffffu, s, off);
        lse_merge(m, s, mo, so);
    }
}

// With LOSS, the row's per-token GRPO loss (token_loss.cuh) is applied to the
// logp just computed, exactly as rk_grpo_token_loss would apply it.
template <bool LOSS>
__global__ void __launch_bounds__(32 * kMergeRowsPerBlock)
    linear_logp_merge(const float2 *__restrict__ part, const float *__restrict__ ztgt,
                      const int64_t *__restrict__ targets, const int32_t *__restrict__ cu,
                      int num_seqs, int64_t T, int32_t V, int32_t num_n, float *__restrict__ logp,
                      float *__restrict__ lse, unsigned *err, GrpoArgs loss) {
    const int64_t row = (int64_t)blockIdx.x * kMergeRowsPerBlock + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= T) return;
    const int64_t tgt = targets[row];
    if (!row_active(row, tgt, cu, num_seqs)) {
        if (lane == 0) {
            logp[row] = 0.f;
            if (lse) lse[row] = 0.f;
            if constexpr (LOSS) grpo_token_inactive(loss, row);
        }
        return;
    }
    if (tgt >= V) {
        if (lane == 0) {
            logp[row] = __int_as_float(0x7fc00000);
            if (lse) lse[row] = __int_as_float(0x7fc00000);
            atomicOr(err, kErrTargetRange);
            if constexpr (LOSS) grpo_token(loss, row, __int_as_float(0x7fc00000));
        }
        return;
    }
    float m, s;
    fold_tiles(part + row * num_n, num_n, lane, m, s);
    if (lane == 0) {
        const float l = __fadd_rn(m, logf(s));
        const float lp = __fsub_rn(ztgt[row], l);
        logp[row] = lp;
        if (lse) lse[row] = l;
        if constexpr (LOSS) grpo_token(loss, row, lp);
    }
}

// Greedy step: the token with the largest logit (lowest index among equal
// maxima; ties across tiles resolve to the lower tile) and its logprob.
__global__ void __launch_bounds__(32 * kMergeRowsPerBlock)
    linear_greedy_merge(const float2 *__restrict__ part, const int32_t *__restrict__ pidx,
                        const int32_t *__restrict__ cu, int num_seqs, int64_t T, int32_t num_n,
                        int64_t *__restrict__ token, float *__restrict__ logp,
                        float *__restrict__ lse) {
    const int64_t row = (int64_t)blockIdx.x * kMergeRowsPerBlock + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= T) return;
    const bool active = cu == nullptr || (row >= (int64_t)cu[0] && row < (int64_t)cu[num_seqs]);
    if (!active) {
        if (lane == 0) {
            token[row] = -1;
            logp[row] = 0.f;
            if (lse) lse[row] = 0.f;
        }
        return;
    }
    float m, s;
    fold_tiles(part + row * num_n, num_n, lane, m, s);
    float bm = -INFINITY;
    int32_t bi = 0x7fffffff;
    for (int j = lane; j < num_n; j += 32) {
        const float x = part[row * num_n + j].x;
        const int32_t i = pidx[row * num_n + j];
        if (x > bm || (x == bm && i < bi)) {
            bm = x;
            bi = i;
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float xo = __shfl_xor_sync(0xffffffffu, bm, off);
        const int32_t io = __shfl_xor_sync(0xffffffffu, bi, off);
        if (xo > bm || (xo == bm && io < bi)) {
            bm = xo;
            bi = io;
        }
    }
    if (lane == 0) {
        const float l = __fadd_rn(m, logf(s));
        token[row] = bi;
        logp[row] = __fsub_rn(bm, l);
        if (lse) lse[row] = l;
    }
}

// Backward rows with a target >= V get NaN gradients (and the error bit).
__global__ void linear_logp_bwd_badtarget(const int64_t *__restrict__ targets,
                                          const int32_t *__restrict__ cu, int num_seqs,
                                          int64_t row0, int64_t rows, int32_t V, int32_t H,
                                          const uint8_t *__restrict__ live,
                                          float *__restrict__ dh, unsigned *err) {
    if ((int64_t)blockIdx.x >= rows) return;
    const int64_t row = row0 + blockIdx.x;
    // live: flags of the blocks of rows [row0, row0 + rows), or null
    if (live != nullptr && live[blockIdx.x / kLiveBlockRows] == 0) {  // a block the dh GEMM skipped
        for (int k = threadIdx.x; k < H; k += blockDim.x) dh[row * H + k] = 0.f;
        return;
    }
    const int64_t tgt = targets[row];
    if (!row_active(row, tgt, cu, num_seqs) || tgt < V) return;
    for (int k = threadIdx.x; k < H; k += blockDim.x) dh[row * H + k] = __int_as_float(0x7fc00000);
    if (threadIdx.x == 0) atomicOr(err, kErrTargetRange);
}

// live[b] = whether any of rows [row0 + 256 b, row0 + 256 b + 256) is active.
__global__ void __launch_bounds__(2 * BM)
    row_blocks_live(const int64_t *__restrict__ targets, const int32_t *__restrict__ cu,
                    int num_seqs, int64_t row0, int64_t rows, uint8_t *__restrict__ live) {
    const int64_t r = (int64_t)blockIdx.x * (2 * BM) + threadIdx.x;
    bool act = false;
    if (r < rows) act = row_active(row0 + r, targets[row0 + r], cu, num_seqs);
    const int any = __syncthreads_or(act ? 1 : 0);
    if (threadIdx.x == 0) live[blockIdx.x] = any != 0 ? 1 : 0;
}

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

template <int MODE>
cudaError_t set_smem_attr(const DeviceInfo &di) {
    static thread_local int done_dev = -1;
    if (done_dev == di.device) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(linear_logp_tiles<MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)TileCfg<MODE>::kSmem);
    if (e == cudaSuccess) done_dev = di.device;
    return e;
}

// CTA pairs that can be resident at once (the persistent grid never exceeds it).
template <int MODE>
int64_t resident_pairs(const DeviceInfo &di) {
    static thread_local int dev = -1;
    static thread_local int64_t val = 0;
    if (dev == di.device) return val;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * (di.sm_count / 2)));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = TileCfg<MODE>::kSmem;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, linear_logp_tiles<MODE>, &cfg) != cudaSuccess || n <= 0) {
        (void)cudaGetLastError();
        n = di.sm_count / 2;
    }
    val = std::min<int64_t>(n, di.sm_count / 2);
    dev = di.device;
    return val;
}

template <int MODE>
cudaError_t run_tiles(const CUtensorMap &tmA, const CUtensorMap &tmB, const TileArgs &a,
                      const DeviceInfo &di, cudaStream_t st, const CUtensorMap *tmC = nullptr,
                      const CUtensorMap *tmD = nullptr) {
    cudaError_t e = set_smem_attr<MODE>(di);
    if (e != cudaSuccess) return e;
    const int64_t tiles =
        (int64_t)((a.num_m + TileCfg<MODE>::kMB - 1) / TileCfg<MODE>::kMB) * a.num_n;
    if (tiles == 0) return cudaSuccess;
    // tile numbers travel as int32 (the queue slots and the counters)
    if (tiles > (int64_t)INT32_MAX) return cudaErrorInvalidValue;
    const int64_t pairs = std::min<int64_t>(tiles, resident_pairs<MODE>(di));
    const unsigned grid = (unsigned)(2 * pairs);
    CUtensorMap unused;
    std::memset(&unused, 0, sizeof(unused));
    if (a.wave_ctr) {
        // rounds: every pair must be resident, so the launch is cooperative
        e = cudaMemsetAsync(a.wave_ctr, 0, sizeof(unsigned), st);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = TileCfg<MODE>::kSmem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, linear_logp_tiles<MODE>, tmA, tmB, tmC ? *tmC : unused,
                                  tmD ? *tmD : unused, a);
    }
    if (a.tile_counter) {
        e = cudaMemsetAsync(a.tile_counter, 0, sizeof(unsigned), st);
        if (e != cudaSuccess) return e;
    }
    linear_logp_tiles<MODE><<<grid, kThreads, TileCfg<MODE>::kSmem, st>>>(
        tmA, tmB, tmC ? *tmC : unused, tmD ? *tmD : unused, a);
    return cudaGetLastError();
}

// The dh / dW GEMMs: two row blocks per tile when the K loop is long (the
// un-overlapped epilogue is then a small part of a tile) and there are enough
// such tiles for about 8 rounds of the resident pairs; one row block per tile
// otherwise.  Either way every accumulator sees the same MMA sequence, so the
// choice does not change any bit.
// A process-wide override (rk_set_row_blocks) can force either form; the
// form each GEMM last used on this host thread is kept for rk_last_row_blocks.
std::atomic<int> g_row_blocks_override{0};
thread_local int g_last_row_blocks[2] = {0, 0};
// Tile order of the last dh / dW GEMM on this host thread: 1 counter, 2 rounds.
thread_local int g_last_tile_order[2] = {0, 0};

template <int M1, int M2>
cudaError_t run_rows(const CUtensorMap &tmA, const CUtensorMap &tmB, const TileArgs &a,
                     const DeviceInfo &di, cudaStream_t st, RowGemm which) {
    const int64_t two = (int64_t)((a.num_m + 1) / 2) * a.num_n;
    const int force = g_row_blocks_override.load(std::memory_order_relaxed);
    const bool use_two =
        force == 2 || (force == 0 && a.num_k >= 256 && two >= 8 * resident_pairs<M2>(di));
    g_last_row_blocks[(int)which] = use_two ? 2 : 1;
    // Long K loops take their tiles in rounds (TileArgs::wave_ctr): pairs
    // that share a dZ row block or a W slice then stay in step, which cut the
    // dh GEMM's DRAM reads at the GRPO size from 115 to 84 GB.  The round
    // counter sits 64 bytes into the launch's 256-byte counter slot.  If the
    // cooperative launch is refused, the tiles come from the counter instead
    // (the order never changes a bit).
    // (Not while the stream is being captured into a graph: there the tiles
    // come from the counter.)
    cudaStreamCaptureStatus capturing = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &capturing) != cudaSuccess) {
        (void)cudaGetLastError();
        capturing = cudaStreamCaptureStatusActive;
    }
    if (a.tile_counter != nullptr && a.num_k >= 256 && capturing == cudaStreamCaptureStatusNone) {
        TileArgs w = a;
        w.wave_ctr = a.tile_counter + 16;
        w.tile_counter = nullptr;
        const cudaError_t e = use_two ? run_tiles<M2>(tmA, tmB, w, di, st)
                                      : run_tiles<M1>(tmA, tmB, w, di, st);
        if (e == cudaSuccess) {
            g_last_tile_order[(int)which] = 2;
            return e;
        }
        (void)cudaGetLastError();
    }
    g_last_tile_order[(int)which] = 1;
    if (use_two) return run_tiles<M2>(tmA, tmB, a, di, st);
    return run_tiles<M1>(tmA, tmB, a, di, st);
}

int64_t ld_dz(int64_t V) { return (V + 7) / 8 * 8; }  // 16-byte aligned dZ rows
int64_t ld_dzt(int64_t n) { return ld_dz(n); }         // dZ^T rows (tokens)

}  // namespace

void set_row_blocks_override(int n) { g_row_blocks_override.store(n, std::memory_order_relaxed); }
int last_row_blocks(RowGemm which) { return g_last_row_blocks[(int)which]; }
int last_tile_order(RowGemm which) { return g_last_tile_order[(int)which]; }

// Every launcher with a workspace keeps the tile counter of its tile
// launches in one 256-byte slot of it.
constexpr size_t kCounterBytes = 256;

// Forward workspace: tile partials [T][num_n], target logits [T], the
// row blocks' live flags [ceil(T / 256)], the tile counter.
size_t linear_fwd_workspace_bytes(int64_t T, int64_t V) {
    if (T <= 0) return 0;
    const int64_t num_n = (V + BN - 1) / BN;
    return round256((size_t)T * (size_t)num_n * sizeof(float2)) + round256((size_t)T * sizeof(float)) +
           round256((size_t)((T + 2 * BM - 1) / (2 * BM))) + kCounterBytes;
}

namespace {
uint8_t *fwd_live_flags(void *workspace, int64_t T, int64_t V) {
    return reinterpret_cast<uint8_t *>(workspace) + linear_fwd_workspace_bytes(T, V) - kCounterBytes -
           round256((size_t)((T + 2 * BM - 1) / (2 * BM)));
}

// Flags the row blocks of [0, T) that hold an active row (the forward's tile
// kernel then skips the others: a padded batch costs no tensor work for its
// padding).
cudaError_t mark_live_blocks(const int64_t *targets, const int32_t *cu, int num_seqs, int64_t T,
                             uint8_t *live, cudaStream_t st) {
    row_blocks_live<<<(unsigned)((T + 2 * BM - 1) / (2 * BM)), 2 * BM, 0, st>>>(targets, cu, num_seqs,
                                                                             0, T, live);
    return cudaGetLastError();
}
}  // namespace

cudaError_t launch_linear_fwd(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                              const int32_t *cu, int num_seqs, int64_t T, int64_t H, int64_t V,
                              float *logp, float *lse, void *workspace, const DeviceInfo &di,
                              cudaStream_t st, const GrpoArgs *loss) {
    if (T == 0) return cudaSuccess;
    CUtensorMap tmA, tmB;
    if (!encode_tmap_bf16_2d(&tmA, h, (uint64_t)H, (uint64_t)T, (uint64_t)H * 2, BK, BM, true))
        return cudaErrorInvalidValue;
    if (!encode_tmap_bf16_2d(&tmB, W, (uint64_t)H, (uint64_t)V, (uint64_t)H * 2, BK, BN / 2, true))
        return cudaErrorInvalidValue;

    TileArgs a{};
    a.targets = targets;
    a.cu = cu;
    a.num_seqs = num_seqs;
    a.row0 = 0;
    a.rows = T;
    a.V = (int32_t)V;
    a.H = (int32_t)H;
    a.num_m = (int32_t)((T + 2 * BM - 1) / (2 * BM));
    a.num_n = (int32_t)((V + BN - 1) / BN);
    a.num_k = (int32_t)(H / BK);
    a.err = di.err;
    a.part = reinterpret_cast<float2 *>(workspace);
    a.ztgt = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(workspace) +
                                       round256((size_t)T * (size_t)a.num_n * sizeof(float2)));
    a.tile_counter = reinterpret_cast<unsigned *>(reinterpret_cast<uint8_t *>(workspace) +
                                                  linear_fwd_workspace_bytes(T, V) - kCounterBytes);
    uint8_t *live = fwd_live_flags(workspace, T, V);
    a.live = live;
    cudaError_t e = mark_live_blocks(targets, cu, num_seqs, T, live, st);
    if (e != cudaSuccess) return e;
    e = run_tiles<kFwd>(tmA, tmB, a, di, st);
    if (e != cudaSuccess) return e;

    const unsigned mgrid = (unsigned)((T + kMergeRowsPerBlock - 1) / kMergeRowsPerBlock);
    if (loss)
        linear_logp_merge<true><<<mgrid, 32 * kMergeRowsPerBlock, 0, st>>>(
            a.part, a.ztgt, targets, cu, num_seqs, T, a.V, a.num_n, logp, lse, di.err, *loss);
    else
        linear_logp_merge<false><<<mgrid, 32 * kMergeRowsPerBlock, 0, st>>>(
            a.part, a.ztgt, targets, cu, num_seqs, T, a.V, a.num_n, logp, lse, di.err, GrpoArgs{});
    return cudaGetLastError();
}

// ---- forward that saves its exponentials, and the backward that uses them ----
// Saved state: the forward workspace (tile partials, target logits, tile
// counter), then e = bf16(2^((z - m_tile) log2 e)) as [T][ld_dz(V)].
size_t linear_fwd_saved_bytes(int64_t T, int64_t V) {
    if (T <= 0) return 0;
    return linear_fwd_workspace_bytes(T, V) + round256((size_t)T * (size_t)ld_dz(V) * 2);
}

cudaError_t launch_linear_fwd_saved(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                                    const int32_t *cu, int num_seqs, int64_t T, int64_t H,
                                    int64_t V, float *logp, float *lse, void *saved,
                                    const DeviceInfo &di, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    CUtensorMap tmA, tmB, tmS;
    if (!encode_tmap_bf16_2d(&tmA, h, (uint64_t)H, (uint64_t)T, (uint64_t)H * 2, BK, BM, true))
        return cudaErrorInvalidValue;
    if (!encode_tmap_bf16_2d(&tmB, W, (uint64_t)H, (uint64_t)V, (uint64_t)H * 2, BK, BN / 2, true))
        return cudaErrorInvalidValue;
    uint8_t *w = reinterpret_cast<uint8_t *>(saved);
    const size_t fwd_bytes = linear_fwd_workspace_bytes(T, V);
    uint16_t *stash = reinterpret_cast<uint16_t *>(w + fwd_bytes);
    if (!encode_tmap_bf16_2d_sw64(&tmS, stash, (uint64_t)V, (uint64_t)T, (uint64_t)ld_dz(V) * 2, 32,
                                  32))
        return cudaErrorInvalidValue;
    TileArgs a{};
    a.targets = targets;
    a.cu = cu;
    a.num_seqs = num_seqs;
    a.row0 = 0;
    a.rows = T;
    a.V = (int32_t)V;
    a.H = (int32_t)H;
    a.num_m = (int32_t)((T + 2 * BM - 1) / (2 * BM));
    a.num_n = (int32_t)((V + BN - 1) / BN);
    a.num_k = (int32_t)(H / BK);
    a.err = di.err;
    a.part = reinterpret_cast<float2 *>(w);
    a.ztgt = reinterpret_cast<float *>(w + round256((size_t)T * (size_t)a.num_n * sizeof(float2)));
    a.tile_counter = reinterpret_cast<unsigned *>(w + fwd_bytes - kCounterBytes);
    uint8_t *live = fwd_live_flags(saved, T, V);
    a.live = live;
    cudaError_t e = mark_live_blocks(targets, cu, num_seqs, T, live, st);
    if (e != cudaSuccess) return e;
    e = run_tiles<kFwdS>(tmA, tmB, a, di, st, nullptr, &tmS);
    if (e != cudaSuccess) return e;
    const unsigned mgrid = (unsigned)((T + kMergeRowsPerBlock - 1) / kMergeRowsPerBlock);
    linear_logp_merge<false><<<mgrid, 32 * kMergeRowsPerBlock, 0, st>>>(
        a.part, a.ztgt, targets, cu, num_seqs, T, a.V, a.num_n, logp, lse, di.err, GrpoArgs{});
    return cudaGetLastError();
}

size_t linear_bwd_saved_workspace_bytes(int64_t T) {
    if (T <= 0) return 0;
    const size_t r = (size_t)T;
    return kCounterBytes + round256(r * 4) + round256(r * (size_t)kEntCap * 8);
}

cudaError_t launch_linear_bwd_saved(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                                    const int32_t *cu, int num_seqs, int64_t T, int64_t H,
                                    int64_t V, const float *lse, const float *grad, void *saved,
                                    float *dh, void *workspace, const DeviceInfo &di,
                                    cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const int64_t ldz = ld_dz(V);
    const int32_t num_n = (int32_t)((V + BN - 1) / BN);
    uint8_t *sv = reinterpret_cast<uint8_t *>(saved);
    const float2 *part = reinterpret_cast<const float2 *>(sv);
    uint16_t *dz = reinterpret_cast<uint16_t *>(sv + linear_fwd_workspace_bytes(T, V));
    // the forward's flags of the row blocks holding an active row: the others
    // are neither converted nor multiplied, and get dh = 0 at the end
    const uint8_t *live = fwd_live_flags(saved, T, V);
    uint8_t *w = reinterpret_cast<uint8_t *>(workspace);
    unsigned *counter = reinterpret_cast<unsigned *>(w);
    int32_t *ecount = reinterpret_cast<int32_t *>(w + kCounterBytes);
    int2 *ent = reinterpret_cast<int2 *>(w + kCounterBytes + round256((size_t)T * 4));

    CUtensorMap tmW_mn;
    if (!encode_tmap_bf16_2d(&tmW_mn, W, (uint64_t)H, (uint64_t)V, (uint64_t)H * 2, 64, BK, true))
        return cudaErrorInvalidValue;
    // dh of rows [r0, r0 + rows) = (the row's fp32 entries) . W - dZ W, K = V
    // in one ascending pass
    auto dh_gemm = [&](int64_t r0, int64_t rows) -> cudaError_t {
        CUtensorMap tmDz;
        if (!encode_tmap_bf16_2d(&tmDz, dz + r0 * ldz, (uint64_t)V, (uint64_t)rows,
                                 (uint64_t)ldz * 2, BK, BM, true))
            return cudaErrorInvalidValue;
        TileArgs a{};
        a.tile_counter = counter;
        a.targets = targets;
        a.cu = cu;
        a.num_seqs = num_seqs;
        a.row0 = r0;
        a.rows = rows;
        a.V = (int32_t)V;
        a.H = (int32_t)H;
        a.err = di.err;
        a.W = W;
        a.dh = dh;
        a.ecount = ecount + r0;
        a.ent = ent + r0 * kEntCap;
        a.live = live + r0 / kLiveBlockRows;  // r0 = 0
        a.num_m = (int32_t)((rows + 2 * BM - 1) / (2 * BM));
        a.num_n = (int32_t)((H + BN - 1) / BN);
        a.num_k = (int32_t)((V + BK - 1) / BK);
        return run_rows<kDh, kDh2>(tmDz, tmW_mn, a, di, st, RowGemm::kDhGemm);
    };
    // the saved terms of rows [r0, r0 + rows) become dZ in place; the target
    // and p >= 1/64 columns become the rows' fp32 entries, weighted from an
    // exact z and sorted by column
    auto convert = [&](int64_t r0, int64_t rows, cudaStream_t s) -> cudaError_t {
        cudaError_t e2 = launch_stash_to_dz(dz, ldz, part, num_n, targets, cu, num_seqs, r0, rows, V,
                                            lse, grad, live, ecount, ent, di, s);
        if (e2 != cudaSuccess) return e2;
        e2 = launch_exact_entries(h, W, H, targets, cu, num_seqs, r0, rows, V, lse, grad, ecount,
                                  ent, s);
        if (e2 != cudaSuccess) return e2;
        return launch_sort_entries(ecount + r0, ent + r0 * kEntCap, rows, s);
    };

    // (Converting one chunk of rows beside the dh GEMM of the previous one, on
    // a second stream, measured no faster: 44.0-44.3 ms against 43.0-43.5 ms
    // for the backward call at the GRPO size, in an A/B on one box.)
    cudaError_t e = cudaMemsetAsync(ecount, 0, (size_t)T * 4, st);
    if (e == cudaSuccess) e = convert(0, T, st);
    if (e == cudaSuccess) e = dh_gemm(0, T);
    if (e != cudaSuccess) return e;
    // rows of the blocks the forward found without an active row: dh = 0
    linear_logp_bwd_badtarget<<<(unsigned)T, 128, 0, st>>>(targets, cu, num_seqs, 0, T, (int32_t)V,
                                                          (int32_t)H, live, dh, di.err);
    return cudaGetLastError();
}

size_t linear_greedy_workspace_bytes(int64_t T, int64_t V) {
    if (T <= 0) return 0;
    const int64_t num_n = (V + BN - 1) / BN;
    return linear_fwd_workspace_bytes(T, V) + round256((size_t)T * (size_t)num_n * sizeof(int32_t));
}

cudaError_t launch_linear_greedy(const uint16_t *h, const uint16_t *W, const int32_t *cu,
                                 int num_seqs, int64_t T, int64_t H, int64_t V, int64_t *token,
                                 float *logp, float *lse, void *workspace, const DeviceInfo &di,
                                 cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    CUtensorMap tmA, tmB;
    if (!encode_tmap_bf16_2d(&tmA, h, (uint64_t)H, (uint64_t)T, (uint64_t)H * 2, BK, BM, true))
        return cudaErrorInvalidValue;
    if (!encode_tmap_bf16_2d(&tmB, W, (uint64_t)H, (uint64_t)V, (uint64_t)H * 2, BK, BN / 2, true))
        return cudaErrorInvalidValue;
    TileArgs a{};
    a.targets = nullptr;
    a.cu = cu;
    a.num_seqs = num_seqs;
    a.row0 = 0;
    a.rows = T;
    a.V = (int32_t)V;
    a.H = (int32_t)H;
    a.num_m = (int32_t)((T + 2 * BM - 1) / (2 * BM));
    a.num_n = (int32_t)((V + BN - 1) / BN);
    a.num_k = (int32_t)(H / BK);
    a.err = di.err;
    uint8_t *w = reinterpret_cast<uint8_t *>(workspace);
    a.part = reinterpret_cast<float2 *>(w);
    const size_t fwd_bytes = linear_fwd_workspace_bytes(T, V);
    a.ztgt = reinterpret_cast<float *>(w + round256((size_t)T * (size_t)a.num_n * sizeof(float2)));
    a.pidx = reinterpret_cast<int32_t *>(w + fwd_bytes);
    a.tile_counter = reinterpret_cast<unsigned *>(w + fwd_bytes - kCounterBytes);
    cudaError_t e = run_tiles<kGreedy>(tmA, tmB, a, di, st);
    if (e != cudaSuccess) return e;
    const unsigned mgrid = (unsigned)((T + kMergeRowsPerBlock - 1) / kMergeRowsPerBlock);
    linear_greedy_merge<<<mgrid, 32 * kMergeRowsPerBlock, 0, st>>>(a.part, a.pidx, cu, num_seqs, T,
                                                                    a.num_n, token, logp, lse);
    return cudaGetLastError();
}

cudaError_t launch_lm_head(const uint16_t *h, const uint16_t *W, int64_t T, int64_t H, int64_t V,
                           uint16_t *logits, int64_t ld, unsigned *tile_counter,
                           const DeviceInfo &di, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    CUtensorMap tmA, tmB;
    if (!encode_tmap_bf16_2d(&tmA, h, (uint64_t)H, (uint64_t)T, (uint64_t)H * 2, BK, BM, true))
        return cudaErrorInvalidValue;
    if (!encode_tmap_bf16_2d(&tmB, W, (uint64_t)H, (uint64_t)V, (uint64_t)H * 2, BK, BN / 2, true))
        return cudaErrorInvalidValue;
    TileArgs a{};
    a.targets = nullptr;
    a.row0 = 0;
    a.rows = T;
    a.V = (int32_t)V;
    a.H = (int32_t)H;
    a.num_m = (int32_t)((T + 2 * BM - 1) / (2 * BM));
    a.num_n = (int32_t)((V + BN - 1) / BN);
    a.num_k = (int32_t)(H / BK);
    a.err = di.err;
    a.dz = logits;
    a.ldz = ld;
    a.tile_counter = tile_counter;  // null: fixed tile lists
    return run_tiles<kLogits>(tmA, tmB, a, di, st);
}

size_t linear_dw_workspace_bytes(int64_t n, int64_t H, int64_t V) {
    if (n <= 0) return 0;
    const size_t ln = (size_t)n;
    size_t b = kCounterBytes;                               // tile counter
    b += round256(ln * 8) + round256(8);                    // crow, n_active
    b += round256(ln * (size_t)H * 2);                      // hc
    b += 2 * round256(ln * 4) + round256(ln * 8);           // gc, lsec, tgtc
    const size_t le = ln * (size_t)kEntCap;                 // entries, at most
    b += round256(ln * 4) + round256(le * 8);               // ecount, ent
    b += round256(ln * 4) + round256(8);                    // eoff, etotal
    b += 2 * round256(le * 4);                              // ent_t, ent_w
    b += 4 * round256(le * 4);                              // sort buffers
    b += 2 * round256((size_t)V * 4);                       // begin, end
    b += round256((size_t)V * 4) + round256(8);             // rows, n_rows
    b += round256((size_t)dw_scan_entries((int64_t)le) * 4);  // scan counts
    // dZ [n][round_up(V, 8)] or dZ^T [V][round_up(n, 8)], whichever is larger
    b += round256(std::max(ln * (size_t)ld_dz(V), (size_t)V * (size_t)ld_dzt(n)) * 2);
    return b;
}

size_t linear_bwd_full_workspace_bytes(int64_t n, int64_t H, int64_t V) {
    if (n <= 0) return 0;
    // the dW buffers plus a dZ^T [V][round_up(n, 8)] next to dZ
    return linear_dw_workspace_bytes(n, H, V) + round256((size_t)V * (size_t)ld_dzt(n) * 2);
}

// Canonical backward: prep + dZ over the canonical tokens, then (if dh) the
// dh GEMM scattered back to physical rows, then (if dW) the dW GEMM.
static cudaError_t canonical_backward(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                                      const int32_t *cu, int num_seqs, int64_t T, int64_t H,
                                      int64_t V, const float *lse, const float *grad,
                                      const int64_t *order, int64_t n, float *dh, float *dW,
                                      void *workspace, const DeviceInfo &di, cudaStream_t st,
                                      const void *saved = nullptr);

cudaError_t launch_linear_dw(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                             const int32_t *cu, int num_seqs, int64_t T, int64_t H, int64_t V,
                             const float *lse, const float *grad, const int64_t *order, int64_t n,
                             float *dW, void *workspace, const DeviceInfo &di, cudaStream_t st) {
    return canonical_backward(h, W, targets, cu, num_seqs, T, H, V, lse, grad, order, n, nullptr,
                              dW, workspace, di, st);
}

cudaError_t launch_linear_bwd_full(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                                   const int32_t *cu, int num_seqs, int64_t T, int64_t H, int64_t V,
                                   const float *lse, const float *grad, const int64_t *order,
                                   int64_t n, float *dh, float *dW, void *workspace,
                                   const DeviceInfo &di, cudaStream_t st, const void *saved) {
    // rows outside the canonical set keep dh = 0; out-of-range targets get NaN
    cudaError_t e = cudaMemsetAsync(dh, 0, (size_t)T * (size_t)H * sizeof(float), st);
    if (e != cudaSuccess) return e;
    e = canonical_backward(h, W, targets, cu, num_seqs, T, H, V, lse, grad, order, n, dh, dW,
                           workspace, di, st, saved);
    if (e != cudaSuccess) return e;
    if (T > 0) {
        linear_logp_bwd_badtarget<<<(unsigned)T, 128, 0, st>>>(
            targets, cu, num_seqs, 0, T, (int32_t)V, (int32_t)H, nullptr, dh, di.err);
        e = cudaGetLastError();
    }
    return e;
}

static cudaError_t canonical_backward(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                                      const int32_t *cu, int num_seqs, int64_t T, int64_t H,
                                      int64_t V, const float *lse, const float *grad,
                                      const int64_t *order, int64_t n, float *dh, float *dW,
                                      void *workspace, const DeviceInfo &di, cudaStream_t st,
                                      const void *saved) {
    if (saved && !dh) return cudaErrorInvalidValue;  // the saved form is the full backward
    if (n == 0)
        return dW ? cudaMemsetAsync(dW, 0, (size_t)V * (size_t)H * sizeof(float), st) : cudaSuccess;
    uint8_t *w = reinterpret_cast<uint8_t *>(workspace);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        uint8_t *p = w + off;
        off += round256(bytes);
        return p;
    };
    const size_t ln = (size_t)n;
    unsigned *counter = reinterpret_cast<unsigned *>(take(kCounterBytes));
    DwBuffers bf;
    bf.crow = reinterpret_cast<int64_t *>(take(ln * 8));
    bf.n_active = reinterpret_cast<int64_t *>(take(8));
    bf.hc = reinterpret_cast<uint16_t *>(take(ln * (size_t)H * 2));
    bf.gc = reinterpret_cast<float *>(take(ln * 4));
    bf.lsec = reinterpret_cast<float *>(take(ln * 4));
    bf.tgtc = reinterpret_cast<int64_t *>(take(ln * 8));
    const size_t le = ln * (size_t)kEntCap;
    bf.ecount = reinterpret_cast<int32_t *>(take(ln * 4));
    bf.ent = reinterpret_cast<int2 *>(take(le * 8));
    bf.eoff = reinterpret_cast<int32_t *>(take(ln * 4));
    bf.etotal = reinterpret_cast<int64_t *>(take(8));
    bf.ent_t = reinterpret_cast<int32_t *>(take(le * 4));
    bf.ent_w = reinterpret_cast<float *>(take(le * 4));
    bf.key0 = reinterpret_cast<int32_t *>(take(le * 4));
    bf.val0 = reinterpret_cast<int32_t *>(take(le * 4));
    bf.key1 = reinterpret_cast<int32_t *>(take(le * 4));
    bf.val1 = reinterpret_cast<int32_t *>(take(le * 4));
    bf.begin = reinterpret_cast<int32_t *>(take((size_t)V * 4));
    bf.end = reinterpret_cast<int32_t *>(take((size_t)V * 4));
    bf.rows = reinterpret_cast<int32_t *>(take((size_t)V * 4));
    bf.n_rows = reinterpret_cast<int64_t *>(take(8));
    bf.scan = reinterpret_cast<int32_t *>(take((size_t)dw_scan_entries((int64_t)le) * 4));
    bf.ldz = ld_dz(V);
    bf.dz = reinterpret_cast<uint16_t *>(
        take(std::max(ln * (size_t)bf.ldz, (size_t)V * (size_t)ld_dzt(n)) * 2));
    // the full backward keeps both dZ (for dh) and dZ^T (for dW)
    uint16_t *dzT = dh ? reinterpret_cast<uint16_t *>(take((size_t)V * (size_t)ld_dzt(n) * 2)) : bf.dz;
    const int64_t ldn = ld_dzt(n);

    cudaError_t e = launch_dw_prep(h, targets, cu, num_seqs, T, H, V, lse, grad, order, n, bf, di, st);
    if (e != cudaSuccess) return e;

    CUtensorMap tmHc, tmW;
    // dW = S - dZ^T h with A = dZ^T read K-major (rows = vocabulary, columns =
    // H, K = canonical tokens), B = h read MN-major; S from the sorted flat
    // list of fp32 entries
    auto run_dw = [&]() -> cudaError_t {
        cudaError_t e2 = launch_dw_entries(n, V, bf, bf.hc, H, dW, di, st);
        if (e2 != cudaSuccess) return e2;
        CUtensorMap tmDzTk, tmHcT2;
        if (!encode_tmap_bf16_2d(&tmDzTk, dzT, (uint64_t)n, (uint64_t)V, (uint64_t)ldn * 2, BK, BM,
                                 true))
            return cudaErrorInvalidValue;
        if (!encode_tmap_bf16_2d(&tmHcT2, bf.hc, (uint64_t)H, (uint64_t)n, (uint64_t)H * 2, 64, BK,
                                 true))
            return cudaErrorInvalidValue;
        TileArgs d{};
        d.tile_counter = counter;
        d.targets = nullptr;
        d.rows = V;
        d.V = (int32_t)V;
        d.H = (int32_t)H;
        d.err = di.err;
        d.dw_begin = bf.begin;
        d.dw_end = bf.end;
        d.dw = dW;
        d.num_m = (int32_t)((V + 2 * BM - 1) / (2 * BM));
        d.num_n = (int32_t)((H + BN - 1) / BN);
        d.num_k = (int32_t)((n + BK - 1) / BK);
        return run_rows<kDwK, kDwK2>(tmDzTk, tmHcT2, d, di, st, RowGemm::kDwGemm);
    };
    if (!dh) {
        // dW alone: dZ^T over the canonical tokens (z^T = W h^T, both operands
        // K-major), then the dW GEMM
        CUtensorMap tmWa, tmHcb;
        if (!encode_tmap_bf16_2d(&tmWa, W, (uint64_t)H, (uint64_t)V, (uint64_t)H * 2, BK, BM, true))
            return cudaErrorInvalidValue;
        if (!encode_tmap_bf16_2d(&tmHcb, bf.hc, (uint64_t)H, (uint64_t)n, (uint64_t)H * 2, BK,
                                 BN / 2, true))
            return cudaErrorInvalidValue;
        TileArgs t{};
        t.tile_counter = counter;
        t.targets = bf.tgtc;  // each token column's target
        t.ecount = bf.ecount;
        t.ent = bf.ent;
        t.rows = V;
        t.V = (int32_t)V;
        t.H = (int32_t)H;
        t.err = di.err;
        t.lse = bf.lsec;
        t.grad = bf.gc;
        t.dz = bf.dz;
        t.ldz = ldn;
        t.ntok = n;
        t.num_m = (int32_t)((V + 2 * BM - 1) / (2 * BM));
        t.num_n = (int32_t)((n + BN - 1) / BN);
        t.num_k = (int32_t)(H / BK);
        CUtensorMap tmDzTs;
        if (!encode_tmap_bf16_2d_sw64(&tmDzTs, dzT, (uint64_t)n, (uint64_t)V, (uint64_t)ldn * 2, 32,
                                      32))
            return cudaErrorInvalidValue;
        t.dz_tma = true;
        e = run_tiles<kDzT>(tmWa, tmHcb, t, di, st, nullptr, &tmDzTs);
        if (e != cudaSuccess) return e;
        return run_dw();
    }

    TileArgs a{};
    a.tile_counter = counter;
    a.targets = bf.tgtc;
    a.cu = nullptr;
    a.num_seqs = 0;
    a.row0 = 0;
    a.rows = n;
    a.V = (int32_t)V;
    a.H = (int32_t)H;
    a.err = di.err;
    a.lse = bf.lsec;
    a.grad = bf.gc;
    a.dz = bf.dz;
    a.ldz = bf.ldz;
    a.ecount = bf.ecount;
    a.ent = bf.ent;
    a.num_m = (int32_t)((n + 2 * BM - 1) / (2 * BM));
    a.num_n = (int32_t)((V + BN - 1) / BN);
    a.num_k = (int32_t)(H / BK);
    if (saved) {
        // dZ over the canonical tokens from the forward's saved terms (the
        // same conversion as rk_linear_logp_bwd_saved, so the same bits), the
        // entries' fp32 weights from an exact z; dZ^T by a transpose
        const uint8_t *sv = reinterpret_cast<const uint8_t *>(saved);
        const float2 *part = reinterpret_cast<const float2 *>(sv);
        const uint16_t *terms = reinterpret_cast<const uint16_t *>(sv + linear_fwd_workspace_bytes(T, V));
        e = launch_stash_to_dz_canonical(terms, bf.ldz, part, (int32_t)((V + BN - 1) / BN), bf.crow,
                                         bf.n_active, bf.tgtc, bf.lsec, bf.gc, n, V, bf.dz,
                                         bf.ecount, bf.ent, di, st);
        if (e != cudaSuccess) return e;
        e = launch_exact_entries(bf.hc, W, H, bf.tgtc, nullptr, 0, 0, n, V, bf.lsec, bf.gc,
                                 bf.ecount, bf.ent, st);
        if (e != cudaSuccess) return e;
        e = launch_transpose_dz(bf.dz, bf.ldz, n, V, dzT, ldn, st);
        if (e != cudaSuccess) return e;
    } else {
        // dZ over the canonical tokens (every position past the active count
        // has target -1 and so gives a zero row), dZ^T as well, through 32 x 32
        // TMA stores from the epilogue
        if (!encode_tmap_bf16_2d(&tmHc, bf.hc, (uint64_t)H, (uint64_t)n, (uint64_t)H * 2, BK, BM,
                                 true))
            return cudaErrorInvalidValue;
        if (!encode_tmap_bf16_2d(&tmW, W, (uint64_t)H, (uint64_t)V, (uint64_t)H * 2, BK, BN / 2,
                                 true))
            return cudaErrorInvalidValue;
        CUtensorMap tmDzTs;
        if (!encode_tmap_bf16_2d(&tmDzTs, dzT, (uint64_t)n, (uint64_t)V, (uint64_t)ldn * 2, 32, 32,
                                 false))
            return cudaErrorInvalidValue;
        CUtensorMap tmDzS;
        if (!encode_tmap_bf16_2d_sw64(&tmDzS, bf.dz, (uint64_t)V, (uint64_t)n, (uint64_t)bf.ldz * 2,
                                      32, 32))
            return cudaErrorInvalidValue;
        a.dzT_store = true;
        a.dz_tma = true;
        e = run_tiles<kDz>(tmHc, tmW, a, di, st, &tmDzTs, &tmDzS);
        if (e != cudaSuccess) return e;
        a.dzT_store = false;
        a.dz_tma = false;
    }

    if (dh) {
        // dh over the canonical rows, K = V ascending, each row stored at its
        // physical position (the same arithmetic per row as rk_linear_logp_bwd)
        e = launch_sort_entries(bf.ecount, bf.ent, n, st);
        if (e != cudaSuccess) return e;
        CUtensorMap tmDz, tmWmn;
        if (!encode_tmap_bf16_2d(&tmDz, bf.dz, (uint64_t)V, (uint64_t)n, (uint64_t)bf.ldz * 2, BK,
                                 BM, true))
            return cudaErrorInvalidValue;
        if (!encode_tmap_bf16_2d(&tmWmn, W, (uint64_t)H, (uint64_t)V, (uint64_t)H * 2, 64, BK, true))
            return cudaErrorInvalidValue;
        TileArgs q = a;
        q.W = W;
        q.dh = dh;
        q.out_rows = bf.crow;
        q.num_n = (int32_t)((H + BN - 1) / BN);
        q.num_k = (int32_t)((V + BK - 1) / BK);
        e = run_rows<kDh, kDh2>(tmDz, tmWmn, q, di, st, RowGemm::kDhGemm);
        if (e != cudaSuccess) return e;
    }
    if (!dW) return cudaSuccess;
    return run_dw();
}

int64_t linear_bwd_chunk_quantum() { return BM; }

// Backward workspace for a chunk of rows: tile counter, the rows' entry
// counts and entry lists, dZ, then the live flags of the chunk's row blocks.
size_t linear_bwd_chunk_bytes(int64_t rows, int64_t V) {
    const size_t r = (size_t)rows;
    return kCounterBytes + round256(r * 4) + round256(r * (size_t)kEntCap * 8) +
           round256(r * (size_t)ld_dz(V) * 2) + round256((r + kLiveBlockRows - 1) / kLiveBlockRows);
}

cudaError_t launch_linear_bwd(const uint16_t *h, const uint16_t *W, const int64_t *targets,
                              const int32_t *cu, int num_seqs, int64_t T, int64_t H, int64_t V,
                              const float *lse, const float *grad, float *dh, void *workspace,
                              size_t workspace_bytes, const DeviceInfo &di, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    const int64_t ldz = ld_dz(V);
    // rows per chunk: as many whole 128-row blocks as the workspace holds
    const size_t per_row = 4 + (size_t)kEntCap * 8 + (size_t)ldz * 2;
    if (workspace_bytes < kCounterBytes) return cudaErrorInvalidValue;
    int64_t chunk = (int64_t)((workspace_bytes - kCounterBytes) / per_row) / BM * BM;
    while (chunk > 0 && linear_bwd_chunk_bytes(chunk, V) > workspace_bytes) chunk -= BM;
    if (chunk <= 0) return cudaErrorInvalidValue;
    if (chunk > T) chunk = T;
    uint8_t *w = reinterpret_cast<uint8_t *>(workspace);
    unsigned *counter = reinterpret_cast<unsigned *>(w);
    int32_t *ecount = reinterpret_cast<int32_t *>(w + kCounterBytes);
    int2 *ent = reinterpret_cast<int2 *>(w + kCounterBytes + round256((size_t)chunk * 4));
    uint16_t *dz = reinterpret_cast<uint16_t *>(w + kCounterBytes + round256((size_t)chunk * 4) +
                                                round256((size_t)chunk * (size_t)kEntCap * 8));
    uint8_t *live = reinterpret_cast<uint8_t *>(dz) + round256((size_t)chunk * (size_t)ldz * 2);

    CUtensorMap tmW_k, tmW_mn;
    if (!encode_tmap_bf16_2d(&tmW_k, W, (uint64_t)H, (uint64_t)V, (uint64_t)H * 2, BK, BN / 2, true))
        return cudaErrorInvalidValue;
    if (!encode_tmap_bf16_2d(&tmW_mn, W, (uint64_t)H, (uint64_t)V, (uint64_t)H * 2, 64, BK, true))
        return cudaErrorInvalidValue;

    for (int64_t r0 = 0; r0 < T; r0 += chunk) {
        const int64_t rows = std::min(chunk, T - r0);
        CUtensorMap tmH, tmDz;
        if (!encode_tmap_bf16_2d(&tmH, h + r0 * H, (uint64_t)H, (uint64_t)rows, (uint64_t)H * 2, BK,
                                 BM, true))
            return cudaErrorInvalidValue;
        if (!encode_tmap_bf16_2d(&tmDz, dz, (uint64_t)V, (uint64_t)rows, (uint64_t)ldz * 2, BK, BM,
                                 true))
            return cudaErrorInvalidValue;

        TileArgs a{};
        a.tile_counter = counter;
        a.targets = targets;
        a.cu = cu;
        a.num_seqs = num_seqs;
        a.row0 = r0;
        a.rows = rows;
        a.V = (int32_t)V;
        a.H = (int32_t)H;
        a.err = di.err;
        a.lse = lse;
        a.grad = grad;
        a.dz = dz;
        a.ldz = ldz;
        a.W = W;
        a.dh = dh;
        a.ecount = ecount;
        a.ent = ent;
        a.num_m = (int32_t)((rows + 2 * BM - 1) / (2 * BM));
        // the chunk's row blocks without an active row: skipped by both GEMMs
        a.live = live;
        row_blocks_live<<<(unsigned)a.num_m, 2 * BM, 0, st>>>(targets, cu, num_seqs, r0, rows, live);

        // GEMM 1: z recomputed, dZ = g exp(z - lse) in bf16 (the target and
        // p >= 1/64 columns as fp32 entries instead), stored by TMA
        cudaError_t e = cudaMemsetAsync(ecount, 0, (size_t)rows * 4, st);
        if (e != cudaSuccess) return e;
        CUtensorMap tmDzS;
        if (!encode_tmap_bf16_2d_sw64(&tmDzS, dz, (uint64_t)V, (uint64_t)rows, (uint64_t)ldz * 2, 32,
                                      32))
            return cudaErrorInvalidValue;
        a.num_n = (int32_t)((V + BN - 1) / BN);
        a.num_k = (int32_t)(H / BK);
        a.dz_tma = true;
        e = run_tiles<kDz>(tmH, tmW_k, a, di, st, nullptr, &tmDzS);
        if (e != cudaSuccess) return e;
        a.dz_tma = false;
        e = launch_sort_entries(ecount, ent, rows, st);
        if (e != cudaSuccess) return e;

        // GEMM 2: dh = (the row's fp32 entries) . W - dZ W, K = V in one
        // ascending pass
        a.num_n = (int32_t)((H + BN - 1) / BN);
        a.num_k = (int32_t)((V + BK - 1) / BK);
        e = run_rows<kDh, kDh2>(tmDz, tmW_mn, a, di, st, RowGemm::kDhGemm);
        if (e != cudaSuccess) return e;
        // out-of-range targets, and dh = 0 on the skipped blocks
        linear_logp_bwd_badtarget<<<(unsigned)rows, 128, 0, st>>>(targets, cu, num_seqs, r0, rows,
                                                                 (int32_t)V, (int32_t)H, live, dh,
                                                                 di.err);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace rk
