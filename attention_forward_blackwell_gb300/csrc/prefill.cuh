// Warp-specialised prefill attention forward for sm_103a.
//
// Method: "b200-flash-attention4-planner".  Section A1 gives the streaming
// online softmax (per key/value block: S = Q K^T, new running max, rebase the
// old row_sum and O, P = exp(S - max), O += P V, divide by row_sum only at the
// end) and the role split (a TMA load warp, an MMA-issuing warp, softmax
// warpgroups for a two-stage Q pipeline, a correction/epilogue warpgroup, a
// store).  Section E steps 3-8 give the two MMAs, the S/P/O regions in tensor
// memory, the barrier graph (Q/K/V ready -> score MMA; S ready -> softmax;
// P ready + O safe -> value MMA; final O -> epilogue -> store), the scalar
// mailbox, the causal block classes (skipped / full / diagonal) and the O
// correction.  The design below is our own for sm_103a:
//
//   CTA = (query block, query head, batch entry).  For head_dim <= 128 a CTA
//   owns two 128-row Q tiles (NQ = 2) that share one K/V stream; for
//   head_dim = 256 it owns one Q tile (NQ = 1) and ping-pongs two score
//   buffers instead, because two 256-column O accumulators do not fit the
//   512 tensor-memory columns.
//
//   warps 0..4*NQ-1   softmax, one warpgroup per Q tile; thread = query row
//                     = tensor-memory lane
//   next warpgroup    correction (rebases O when the running max jumps) and
//                     epilogue (O / row_sum -> bf16 -> smem -> TMA store; LSE)
//   next warp         tcgen05.mma issue (one elected lane)
//   next warp         TMA producer (Q once, then K_j, V_j through the ring)
//
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   NQ = 2: S_t at columns [128 t, 128 t + 128), O_t at [256 + 128 t, ...).
//           P_t (bf16 pairs) overwrites the upper half of S_t.
//   NQ = 1: S buffers at [0, 128) and [128, 256), O at [256, 512).
//
// Hazard on the P/S alias: the next score MMA S_t(j+1) overwrites the upper
// half of S_t, i.e. P_t(j), which the value MMA PV_t(j) reads.  MMAs with
// different accumulators are not ordered by the ISA, so the MMA warp issues
// S_t(j+1) only once PV_t(j) has completed (tcgen05.commit -> mbarrier); the
// tensor core is busy with that PV while the warp waits.  Descriptors are
// built once per CTA as their lower 32-bit words and advanced by address
// offsets, so each MMA issue is one add per operand and the instruction
// itself (the issuing thread's instruction count sets the pace).
//
// Work split: one CTA per unit; when the units do not fill the last wave,
// those of the last partial wave are cut along the key axis into pieces that
// write unnormalised partial results, and the last piece to arrive merges
// them on all threads of its CTA after its roles finish (merge_unit).
//
// Rebasing: the running max m is only moved when the block max exceeds it by
// more than kRescaleThreshold (log2 units).  Until then P = exp2(s - m) may
// exceed 1 by at most 2^threshold, which fp32 accumulates exactly as well;
// O / row_sum and LSE = m + log2(row_sum) are unchanged by the choice of m.
// When m moves, both row_sum and O are multiplied by exp2(m_old - m_new), as
// the streaming recurrence requires.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace fa {

constexpr float kRescaleThreshold = 8.0f;   // log2 units (a factor of 256)


// Optionally (kUsePolyExp2), in tiles without masked entries one pair of
// exponentials in every kPolyEvery is computed by exp2_poly_x2 on the FMA
// pipe instead of the MUFU ex2 instruction.  Measured on GB300 this is slower
// at head_dim 128 (the softmax is bound by instruction issue, not by the MUFU
// pipe), so it is off.
constexpr bool kUsePolyExp2 = false;
constexpr int kPolyEvery = 4;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

template <int D>
struct PrefillTraits {
    static constexpr int BM = 128;                     // rows per Q tile = TMEM lanes
    static constexpr int BN = 128;                     // keys per K/V tile
    static constexpr int NQ = (D <= 128) ? 2 : 1;      // Q tiles per CTA
    static constexpr int NSBUF = (NQ == 2) ? 1 : 2;    // score buffers per Q tile
    static constexpr int NCH = (D + 63) / 64;          // 64-element (128-byte) row chunks
    static constexpr int CHUNK = 128 * 128;            // one chunk of 128 rows, bytes
    static constexpr int QTILE = NCH * CHUNK;
    // head_dim 512: the output columns are shared out over DV_SPLIT = 2 CTAs
    // per Q tile (each computes the full scores and one 256-column half of
    // O), because 512 fp32 O columns leave no tensor memory for the scores.
    static constexpr int DV_SPLIT = (D == 512) ? 2 : 1;
    static constexpr int D_COLS = D / DV_SPLIT;        // O accumulator columns of a CTA
    // One Q tile (head_dim >= 256): the ring is filled in the order the MMA
    // warp consumes it (K_0, then K_{j+1} before V_j) and each slot is
    // released as soon as the MMAs that read it complete.
    static constexpr bool CONSUME_ORDER = (D >= 256);
    // head_dim 256: the Q, K and V tensor maps are 4-D, {64 columns, rows,
    // 64-column chunks, planes} with a chunk stride of 128 bytes, and one
    // copy brings a {64, 128, 2, 1} box: two chunks (32 KB) written as
    // [chunk][row][64 columns], the layout of two 3-D boxes.  The SM's copy
    // engine spends about as long on a box of 2 x 128 rows as on one of 128
    // rows (measured on GB300: ~350 vs ~235 cycles at full occupancy), which
    // matters where a key block brings 128 KB.  (At head_dim 128 the same
    // boxes measured 1 % slower; head_dim 96 cannot use them: its second
    // chunk is half a row, and a 4-D box would read the next row's first
    // columns into it, past the tensor at its last row.)
    static constexpr bool BOX4 = (D == 256);
    static constexpr int OCH = (D_COLS + 63) / 64;     // 64-column chunks of a CTA's O
    // Epilogue: the softmax warpgroup of a tile, idle once its last block is
    // done, stages and stores the first EPI_SPLIT 64-column chunks of that
    // tile's O while the correction warpgroup does the rest (and the LSE),
    // so that the drain of O from tensor memory runs on two warpgroups.
    // Used by the kernels where it measured faster on GB300 (see epi_split).
    static constexpr int EPI_SPLIT = OCH / 2;
    // chunks per ring slot: one at head_dim 512 (the 128 KB Q tile leaves
    // room for five 16 KB slots only)
    static constexpr int SLOT_CH = (D == 512) ? 1 : ((NCH >= 2) ? 2 : 1);
    static constexpr int PIECES = NCH / SLOT_CH;       // ring slots per K tile
    static constexpr int VPIECES = OCH / SLOT_CH;      // ring slots per (own part of a) V tile
    static constexpr int SLOT = SLOT_CH * CHUNK;
    static constexpr int NSLOT = (D == 64) ? 8 : ((D == 512) ? 5 : 4);
    static constexpr int KSTEPS = D / 16;              // score MMA steps of K = 16
    // Value MMA N per instruction (head_dim 96: N = 96, i.e. one full and one
    // half 64-column chunk of the MN-major V tile; head_dim 512: one 64-column
    // chunk, the content of one ring slot; head_dim 256 and 512: all 256
    // columns of the CTA's O).  Measured on GB300: an M = 128, K = 16
    // instruction occupies the tensor pipe ~80 cycles for any N up to 128
    // and 128 cycles at N = 256, so only N = 256 runs at the full rate.
    static constexpr int PV_N = (D <= 128) ? D : 256;
    // head_dim 256 / 512: a V tile (the CTA's 256 columns of it) travels as
    // ring slots of VROW_KEYS keys x 256 columns (four 64-column chunks of
    // VROW_KEYS rows, VROW_CHUNK bytes apart: 64 keys in 32 KB slots at 256,
    // 32 keys in 16 KB slots at 512) instead of slots of 128 keys x 128 or
    // 64 columns, so that each N = 256 value MMA reads one slot, a slot is
    // released after its K-steps, and the value MMA starts once the first
    // slot has landed.
    static constexpr bool VROWS = (D >= 256);
    static constexpr int VROW_KEYS = (D == 512) ? 32 : 64;
    static constexpr int VROW_CHUNK = VROW_KEYS * 128;   // one chunk of VROW_KEYS rows, bytes
    static constexpr int NUM_WARPS = (NQ + 2) * 4;
    static constexpr int THREADS = NUM_WARPS * 32;
    static constexpr int CORR_WG = NQ;
    static constexpr int MMA_WARP = (NQ + 1) * 4;
    static constexpr int LOAD_WARP = MMA_WARP + 1;
    static constexpr uint32_t TMEM_COLS = 512;
    // Register split (threads x registers after setmaxnreg must not exceed
    // the launch allocation: 512 x 128 for NQ = 2, 384 x 168 for NQ = 1).
    // Every target differs from the launch count (increase or decrease).
    // NQ = 2 has two splits, chosen per kernel by measurement on GB300: the
    // kernels with masked scores (causal or windowed) run fastest with
    // 176 / 88 / 72 (no spills; the MMA-issue and TMA warps need under 72),
    // the unmasked one with 168 / 96 / 80.
    static constexpr uint32_t LAUNCH_REGS = (NQ == 2) ? 128 : 168;
    template <bool MASKED>
    struct Regs {
        static constexpr uint32_t SOFTMAX = (NQ == 2) ? (MASKED ? 176 : 168) : 240;
        static constexpr uint32_t CORR = (NQ == 2 && !MASKED) ? 96 : 88;
        static constexpr uint32_t OTHER = (NQ == 2) ? (MASKED ? 72 : 80) : 80;
        static_assert(SOFTMAX > LAUNCH_REGS && CORR < LAUNCH_REGS && OTHER < LAUNCH_REGS,
                      "setmaxnreg targets must move away from the launch allocation");
        static_assert(4 * NQ * 32 * SOFTMAX + 4 * 32 * CORR + 4 * 32 * OTHER <=
                          (NQ + 2) * 128 * LAUNCH_REGS,
                      "register split exceeds the launch allocation");
    };
    static constexpr int SMEM_Q = NQ * QTILE;
    static constexpr int SMEM_RING = NSLOT * SLOT;
    static constexpr int SMEM_AUX = 8192;   // barriers + mailboxes (checked below)
    // head_dim 256 (persistent kernel): STAGE_BUFS 2 KB O staging buffers
    // for each of the correction warps (epilogue stores, see
    // store_o_rows_staged)
    static constexpr int STAGE_BUFS = 3;
    static constexpr int SMEM_STAGE = (D == 256) ? 4 * STAGE_BUFS * 2048 : 0;
    static constexpr int SMEM_TOTAL = 1024 + SMEM_Q + SMEM_RING + SMEM_AUX + SMEM_STAGE;
    static_assert(DV_SPLIT == 1 ? VPIECES == PIECES : NQ == 1,
                  "split output columns only with one Q tile per CTA");
    static_assert(SMEM_TOTAL <= 232448, "shared memory per CTA exceeds the sm_103 limit");
    static_assert(!VROWS || (4 * VROW_CHUNK == SLOT && VPIECES * VROW_KEYS == BN &&
                             D_COLS == 256),
                  "a row-split V slot holds VROW_KEYS keys of the CTA's 256 columns");

    __device__ static constexpr uint32_t s_col(int i) { return (uint32_t)(i * 128); }
    __device__ static constexpr uint32_t o_col(int t) {
        return (NQ == 2) ? (uint32_t)(256 + t * 128) : 256u;
    }
    // head_dim 64: O_t takes 64 of its 128 columns, so P_t (64 columns of
    // bf16 pairs) gets the other 64 instead of the upper half of S_t.  The
    // score MMA of block j+1 then only waits for the softmax to have read
    // S_t(j) (P-ready), not for the value MMA of block j, which runs after
    // it; the softmax waits for that value MMA before it overwrites P_t.
    static constexpr bool SEP_P = (D == 64);
    __device__ static constexpr uint32_t p_col(int t) {
        return SEP_P ? o_col(t) + 64u : s_col(t) + 64u;
    }
    static_assert(!SEP_P || (NQ == 2 && D_COLS <= 64), "separate P columns need room beside O");
};

template <class T>
struct PrefillAux {
    uint64_t bar_q;
    uint64_t bar_full[T::NSLOT];
    uint64_t bar_empty[T::NSLOT];
    uint64_t bar_s_full[2];        // NQ = 2: per tile; NQ = 1: per score buffer
    // P ready + O rebased and the rebase mailbox come in two copies, used by
    // tile (NQ = 2) or by key-block parity (NQ = 1); see sig_idx.
    uint64_t bar_p_ready[2];       // P(j) written and O rebased (softmax + correction)
    uint64_t bar_pv_done[2];       // value MMA completed (copies as for P-ready)
    uint64_t bar_mb_full[2];       // mailbox message j (alpha) posted
    uint64_t bar_fin[T::NQ];       // final row statistics posted (own barrier: the
                                   // final message does not wait for message nk-1
                                   // to be consumed, so sharing mb_full could let
                                   // it complete two phases ahead of its reader)
    uint64_t bar_epi[T::NQ];       // staging of O_t in shared memory complete
    uint64_t bar_epi_sm[T::NQ];    // the softmax warpgroup's part of that staging complete
    uint64_t bar_drain[2];
    uint64_t bar_tail;             // producer-private: partial last value tile landed
    uint64_t bar_split_a;          // piece of a split unit: partial result written (4 warps)
    uint64_t bar_qfree;            // persistent: the unit's last score MMA completed (Q free)
    uint64_t bar_odrained;         // persistent: the unit's O has been read out of tensor memory
    uint32_t tmem_base;
    int abort_flag;
    int merge_last;
    int merge_unit[4];             // tail, head, batch entry, first row of the unit to merge
    float mb_alpha[2][128];
    float mb_l[T::NQ][128];
    float mb_m[T::NQ][128];
};

// Wait-site codes (recorded with kErrWaitTimeout on a time-out).
enum : unsigned int {
    kSiteLoadEmpty = 1, kSiteMmaQ, kSiteMmaK, kSiteMmaV, kSiteMmaP, kSiteLoadTail, kSiteMmaPv,
    kSiteSmS, kSiteSmMbox, kSiteCorrMbox, kSiteCorrPv, kSiteEpiMbox, kSiteEpiPv,
    kSiteEpiStage, kSiteSplitA, kSiteLoadQfree, kSiteMmaOdrained, kSiteSmOdrained, kSiteSmPv,
    kSiteSmXm, kSiteMmaSfree
};

// Recorded if a piece's arrival could not be counted (never expected: every
// failed compare-and-swap means another piece of the unit was counted).
constexpr unsigned int kErrSplitCount = 0x2001u;

// Debug trace stamp (SM clock) by the calling thread, if tracing this CTA.
// Compiled in only with FA_PREFILL_TRACE=1 (otherwise the trace pointer is
// dead code and occupies no registers).
__device__ __forceinline__ void trace_mark(unsigned long long* tr, int role, int j, int e) {
    if (FA_PREFILL_TRACE && tr != nullptr && j * kTraceEvents + e < kTraceSlots)
        tr[role * kTraceSlots + j * kTraceEvents + e] = (unsigned long long)clock64();
}

// Debug trace stamp by the first thread of the calling warpgroup, for code
// that has no trace pointer of its own (compiled in only with
// FA_PREFILL_TRACE=1).
__device__ __forceinline__ void trace_wg(const PrefillArgs& a, int role, int j, int e) {
    if (FA_PREFILL_TRACE && a.trace != nullptr && (int)blockIdx.x == a.trace_block &&
        (threadIdx.x & 127) == 0 && j * kTraceEvents + e < kTraceSlots)
        a.trace[role * kTraceSlots + j * kTraceEvents + e] = (unsigned long long)clock64();
}

// Per-CTA work coordinates, computed identically by every thread.
//
// The grid is one-dimensional.  With output columns split over DV_SPLIT CTAs
// (head_dim 512), the CTA index's fastest digit selects the column part and
// the rest is the unit index below (the parts of one unit run side by side
// and share its Q, K and V through L2).  Its first n_full CTAs each process a whole
// unit (batch entry, query head, query block), in the order query block
// (fastest), head, batch entry; causal units in the order (batch entry, head)
// fastest, then query block heaviest first.  The remaining
// units (the last, partial wave of a grid of whole units) are each split
// along the key axis into `split` pieces of consecutive key blocks, one CTA
// per piece, so that the last wave is `split` times shorter; the pieces write
// partial results and the last one to finish merges them (merge_unit).
// Key-block counters below are local to the CTA's piece: block j of the
// piece is key block kb + j.
struct PrefillWork {
    int b, h, hk, row0, L, off;
    int n_kv[2];   // key blocks of this piece visited by Q tile 0 / 1
    int n_max;
    int kb;        // first key block of the piece (0 for a whole unit)
    int piece;     // -1 for a whole unit, else the piece's scratch slot
    int tail;      // tail unit of the piece (its merge counter)
    // packed sequences only: query rows of the sequence, and its first query
    // token and first key token in the packed tensors
    int Lq, q0, k0;
    int dv0;       // first output column of this CTA (0 unless DV_SPLIT > 1)
};

template <class T, bool CAUSAL, bool WINDOW, bool VARLEN>
__device__ __forceinline__ PrefillWork prefill_work(const PrefillArgs& a, int c) {
    PrefillWork w;
    w.dv0 = 0;
    if constexpr (T::DV_SPLIT > 1) {
        w.dv0 = (c % T::DV_SPLIT) * T::D_COLS;
        c /= T::DV_SPLIT;
    }
    int u, ke;
    if (c < a.n_full) {
        u = c;
        w.kb = 0;
        ke = 0x7fffffff;
        w.piece = -1;
        w.tail = -1;
    } else {
        const int q = c - a.n_full;
        const int k = q % a.split;
        w.tail = q / a.split;
        u = a.n_full + w.tail;
        w.kb = (int)((long long)k * a.nk / a.split);
        ke = (int)((long long)(k + 1) * a.nk / a.split);
        w.piece = q;
    }
    // Causal: query block slowest, heaviest first over every (batch, head), so
    // that the hardware's in-order dispatch to free SMs is a longest-first
    // schedule.  Non-causal units are equal: query block fastest, so that the
    // CTAs running at once share the K/V of few heads in L2.
    const int nbh = a.B * a.Hq;
    const int x = CAUSAL ? u / nbh : u % a.num_mblk;
    const int hb = CAUSAL ? u % nbh : u / a.num_mblk;
    const int mblk = CAUSAL ? (a.num_mblk - 1 - x) : x;
    w.h = hb % a.Hq;
    w.b = hb / a.Hq;
    w.hk = w.h / a.group;
    int L = a.Sk;
    if constexpr (VARLEN) {
        // sequence b's tokens, clamped so that malformed offsets stay inside
        // the packed tensors
        const int qs = min(max(a.cu_seqlens_q[w.b], 0), a.total_q);
        const int qe = min(max(a.cu_seqlens_q[w.b + 1], qs), a.total_q);
        w.q0 = qs;
        w.Lq = qe - qs;
        if (a.block_table != nullptr) {
            // keys in paged caches: per-sequence lengths, rows by page
            L = max(0, min(a.seqlens_k[w.b], a.Sk));
            w.k0 = 0;
        } else {
            const int ks = min(max(a.cu_seqlens_k[w.b], 0), a.total_k);
            const int ke = min(max(a.cu_seqlens_k[w.b + 1], ks), a.total_k);
            w.k0 = ks;
            L = ke - ks;
        }
        w.off = L - w.Lq;
    } else {
        // (Lq, q0, k0 are read by the packed-sequence kernels only)
        if (a.seqlens_k != nullptr) L = max(0, min(a.seqlens_k[w.b], a.Sk));
        w.off = L - a.Sq;
    }
    w.L = L;
    w.row0 = mblk * T::NQ * T::BM;
    if (WINDOW && a.window > 0) {
        // no row of the unit sees a key below its first row's window
        const int lo_min = w.row0 + w.off - a.window + 1;
        if (lo_min > 0) w.kb = max(w.kb, lo_min / T::BN);
    }
    w.n_kv[0] = w.n_kv[1] = 0;
#pragma unroll
    for (int t = 0; t < T::NQ; ++t) {
        int last = L - 1;   // last key any row of the tile can see
        if (CAUSAL) last = min(last, w.row0 + (t + 1) * T::BM - 1 + w.off);
        const int n = last >= 0 ? last / T::BN + 1 : 0;
        const int cnt = min(n, ke) - w.kb;
        w.n_kv[t] = cnt > 0 ? cnt : 0;
        // a tile past the end of its sequence has nothing to compute
        if (VARLEN && w.row0 + t * T::BM >= w.Lq) w.n_kv[t] = 0;
    }
    w.n_max = max(w.n_kv[0], w.n_kv[T::NQ - 1]);
    return w;
}

template <class T, bool CAUSAL, bool WINDOW, bool VARLEN>
__device__ __forceinline__ void prefetch_q_of(const CUtensorMap* tm_q, const PrefillArgs& a,
                                              int c2) {
    const PrefillWork w2 = prefill_work<T, CAUSAL, WINDOW, VARLEN>(a, c2);
    if (w2.n_max <= 0) return;
#pragma unroll
    for (int t = 0; t < T::NQ; ++t) {
        const int row = (VARLEN ? w2.q0 : 0) + w2.row0 + t * T::BM;
        const int plane = VARLEN ? w2.h : w2.b * a.Hq + w2.h;
        if constexpr (T::BOX4) {
#pragma unroll
            for (int c = 0; c < T::NCH; c += 2) tma_prefetch_l2_4d(tm_q, 0, row, c, plane);
        } else {
#pragma unroll
            for (int c = 0; c < T::NCH; ++c) tma_prefetch_l2_3d(tm_q, c * 64, row, plane);
        }
    }
}

// Copy of the P-ready barrier, rebase mailbox and value-MMA completion
// barrier that tile t's key block j uses, and the phase parity of that block
// on it.  With two Q tiles (NQ = 2)
// each tile has its own copy and every block is a phase: S_t(j+1) is issued
// only after PV_t(j), so a tile's softmax never runs a block ahead of its
// correction.  With one tile and two score buffers (NQ = 1) S(j+1) is issued
// before PV(j), so the softmax can finish block j+1 before the correction has
// handled block j; consecutive blocks then alternate between the two copies,
// so that their arrivals and messages never share one (S(j+2) waits for
// PV(j), hence for the correction's handling of block j).  The same holds for
// the completion of value MMAs: a parity wait is exact only while its barrier
// is at most one phase behind, and with NQ = 1 two value MMAs can be in
// flight; on alternating copies the previous PV of a copy (PV(j-2)) has
// always been waited for by the time PV(j) is (S(j) waits for PV(j-2)).
template <class T>
__device__ __forceinline__ int sig_idx(int t, int j) { return T::NQ == 2 ? t : (j & 1); }
template <class T>
__device__ __forceinline__ uint32_t sig_par(int j) {
    return T::NQ == 2 ? (uint32_t)(j & 1) : (uint32_t)((j >> 1) & 1);
}

// Ring position p (K_j piece c at p = 2 j PIECES + c, V_j at (2 j + 1) PIECES + c).
template <class T>
__device__ __forceinline__ uint32_t ring_slot(int p) { return (uint32_t)(p % T::NSLOT); }
template <class T>
__device__ __forceinline__ uint32_t ring_phase(int p) { return (uint32_t)((p / T::NSLOT) & 1); }

// L2 prefetch of the Q tiles of the unit that CTA c2 (a later CTA of the
// grid) will process; issued by the producer lane after its own first loads.
template <class T, bool CAUSAL, bool WINDOW, bool VARLEN>
__device__ __forceinline__ void prefetch_q_of(const CUtensorMap* tm_q, const PrefillArgs& a,
                                              int c2);

// Loads N consecutive 64-column chunks, starting at chunk c0, of the
// 128-row tile at (row, plane) into consecutive CHUNK-byte buffers at dst
// (4-D maps: two chunks per copy; 3-D maps: one).  Issued by one lane.
template <class T, int N>
__device__ __forceinline__ void load_chunks(uint32_t dst, const CUtensorMap* m, int c0, int row,
                                            int plane, uint32_t bar) {
    if constexpr (T::BOX4) {
        static_assert(N % 2 == 0, "4-D boxes carry two chunks");
#pragma unroll
        for (int c = 0; c < N; c += 2)
            tma_load_4d(dst + c * T::CHUNK, m, 0, row, c0 + c, plane, bar);
    } else {
#pragma unroll
        for (int c = 0; c < N; ++c) tma_load_3d(dst + c * T::CHUNK, m, (c0 + c) * 64, row, plane, bar);
    }
}

// Zeroes rows [rv, BN) of every 64-column chunk of one ring slot (all 32
// lanes of the calling warp), then makes the writes visible to the tensor
// core (async proxy).
template <class T>
__device__ __forceinline__ void zero_value_tail(uint32_t slot_addr, int rv) {
    const int lane = threadIdx.x & 31;
    const int granules = (T::BN - rv) * 8;   // 16-byte granules per chunk
#pragma unroll
    for (int c = 0; c < T::SLOT_CH; ++c) {
        const uint32_t base = slot_addr + c * T::CHUNK + rv * 128;
        for (int g = lane; g < granules; g += 32)
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(base + g * 16), "r"(0)
                         : "memory");
    }
    fence_proxy_async_smem();
    __syncwarp();
}

// Row-split value slot (VROWS): zeroes local rows [r0, VROW_KEYS) of each of
// the four chunks, then makes the writes visible to the tensor core.
template <class T>
__device__ __forceinline__ void zero_value_rows(uint32_t slot_addr, int r0) {
    const int lane = threadIdx.x & 31;
    const int granules = (T::VROW_KEYS - r0) * 8;   // 16-byte granules per chunk
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t base = slot_addr + c * T::VROW_CHUNK + r0 * 128;
        for (int g = lane; g < granules; g += 32)
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(base + g * 16), "r"(0)
                         : "memory");
    }
    fence_proxy_async_smem();
    __syncwarp();
}

// ------------------------------------------------------------ producer ----

template <class T, bool CAUSAL, bool WINDOW, bool VARLEN>
__device__ void prefill_load_role(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                  const CUtensorMap* tm_v, const PrefillArgs& a,
                                  const PrefillWork& w, PrefillAux<T>* aux, uint32_t sQ,
                                  uint32_t sRing, const WaitCtx& wc, unsigned long long* tr) {
    const int lane = threadIdx.x & 31;
    if (lane != 0) tr = nullptr;
    if (w.n_max <= 0) return;
    const uint32_t bar_q = smem_u32(&aux->bar_q);
    if (lane == 0) {
        tma_prefetch_desc(tm_q);
        tma_prefetch_desc(tm_k);
        tma_prefetch_desc(tm_v);
        mbar_arrive_expect_tx(bar_q, (uint32_t)(T::NQ * T::QTILE));
#pragma unroll
        for (int t = 0; t < T::NQ; ++t)
            load_chunks<T, T::NCH>(sQ + t * T::QTILE, tm_q, 0,
                                   (VARLEN ? w.q0 : 0) + w.row0 + t * T::BM,
                                   VARLEN ? w.h : w.b * a.Hq + w.h, bar_q);
    }
    // tile coordinates of key block jk: contiguous K/V, or a page of the
    // paged caches (packed sequences: token k0 + row of head hk)
    auto coords = [&](int jk, int& ty, int& tz) {
        ty = (VARLEN ? w.k0 : 0) + jk * T::BN;
        tz = VARLEN ? w.hk : w.b * a.Hkv + w.hk;
        if (a.block_table != nullptr) {
            const int page = a.block_table[(size_t)w.b * a.max_pages + ty / a.page_size];
            ty = ty % a.page_size;
            tz = page * a.Hkv + w.hk;   // out-of-range pages read as zeros (TMA bounds)
        }
    };
    int issued = 0;
    const int total = 2 * w.n_max * T::PIECES;
    for (int p = 0; p < total; ++p) {
        const int j = p / (2 * T::PIECES);
        const int kv = (p / T::PIECES) & 1;
        const int pc = p % T::PIECES;
        const uint32_t slot = ring_slot<T>(p);
        if (!mbar_wait(smem_u32(&aux->bar_empty[slot]), ring_phase<T>(p) ^ 1u, wc,
                       kErrWaitTimeout | kSiteLoadEmpty))
            break;
        trace_mark(tr, kTrLoad, p >> 3, p & 7);
        const uint32_t full = smem_u32(&aux->bar_full[slot]);
        const int jk = w.kb + j;          // key block
        const int rv = w.L - jk * T::BN;  // valid rows of this tile
        int ty, tz;
        coords(jk, ty, tz);
        if (kv == 1 && j == w.n_max - 1 && rv < T::BN) {
            // Partial last value tile: rows [rv, BN) may hold anything (and a
            // zero probability times a non-finite value would poison O), so
            // they are zeroed before the tile is published to the MMA warps.
            const uint32_t tail = smem_u32(&aux->bar_tail);
            if (lane == 0) {
                mbar_arrive_expect_tx(tail, (uint32_t)T::SLOT);
                load_chunks<T, T::SLOT_CH>(sRing + slot * T::SLOT, tm_v, pc * T::SLOT_CH, ty, tz,
                                           tail);
            }
            if (!mbar_wait(tail, (uint32_t)(pc & 1), wc, kErrWaitTimeout | kSiteLoadTail)) break;
            zero_value_tail<T>(sRing + slot * T::SLOT, rv);
            if (lane == 0) mbar_arrive(full);
        } else if (lane == 0) {
            mbar_arrive_expect_tx(full, (uint32_t)T::SLOT);
            load_chunks<T, T::SLOT_CH>(sRing + slot * T::SLOT, kv ? tm_v : tm_k, pc * T::SLOT_CH,
                                       ty, tz, full);
        }
        __syncwarp();
        issued = p + 1;
        if (p == 1 && lane == 0 && a.q_prefetch > 0 &&
            (int)blockIdx.x + a.q_prefetch < (int)gridDim.x)
            prefetch_q_of<T, CAUSAL, WINDOW, VARLEN>(tm_q, a, (int)blockIdx.x + a.q_prefetch);
    }
    // Drain: every copy issued by this warp must have landed before the CTA
    // exits (on the normal path they all have; after an abort some may not).
    if (lane == 0) {
        mbar_wait_drain(bar_q, 0, a.wait_limit_ns);
        const int first = issued > T::NSLOT ? issued - T::NSLOT : 0;
        for (int p = first; p < issued; ++p)
            mbar_wait_drain(smem_u32(&aux->bar_full[ring_slot<T>(p)]), ring_phase<T>(p),
                            a.wait_limit_ns);
    }
    __syncwarp();
}

// ----------------------------------------------------------- MMA issue ----

// Descriptor address offset (bytes >> 4) of K-step kk inside a K-major
// operand stored as 64-column chunks of 128 rows: chunk kk/4, then 32 bytes
// per step inside the 128-byte swizzled row.
__device__ __forceinline__ constexpr uint32_t kstep_off(int kk) {
    return (uint32_t)(((kk >> 2) * 128 * 128 + (kk & 3) * 32) >> 4);
}

// Score MMA S[128 x 128] = Q_t K_j^T: one N = 128 instruction per K-step of
// 16 head dims.  qd: descriptor of the Q tile; kd[p]: descriptors of the ring
// slots that hold the K tile (two slots for head_dim 256).  Descriptors are
// passed as their lower 32-bit words (sdesc_lo_sw128): one add per operand
// per instruction on the issuing thread, and half the registers.
template <class T>
__device__ __forceinline__ void issue_score(uint32_t tmem_d, uint32_t qd,
                                            const uint32_t (&kd)[T::PIECES], uint32_t idesc) {
#pragma unroll
    for (int kk = 0; kk < T::KSTEPS; ++kk) {
        const int piece = kk / (T::SLOT_CH * 4);
        const int kin = kk % (T::SLOT_CH * 4);
        umma_ss_lo(tmem_d, qd + kstep_off(kk), kd[piece] + kstep_off(kin), idesc, kk > 0 ? 1u : 0u);
    }
}

// Value MMA O[:, 0:N] (+)= P V over 128 keys: 8 steps of 16 keys.  V is
// MN-major: 16 keys are two 8-row swizzle atoms, 2048 bytes per step.
template <class T>
__device__ __forceinline__ void issue_value(uint32_t tmem_o, uint32_t tmem_p, uint32_t vd,
                                            uint32_t idesc, bool first) {
#pragma unroll
    for (int kk = 0; kk < T::BN / 16; ++kk)
        umma_ts_lo(tmem_o, tmem_p + kk * 8, vd + (uint32_t)((kk * 2048) >> 4), idesc,
                   (!first || kk > 0) ? 1u : 0u);
}

// Value MMA over a row-split V slot (VROWS): keys [VROW_KEYS h, +VROW_KEYS)
// of the block, all PV_N output columns, steps of 16 keys; the slot holds
// four chunks (VROW_CHUNK apart, the descriptor's leading byte offset),
// 2048 bytes per step.
template <class T>
__device__ __forceinline__ void issue_value_rows(uint32_t tmem_o, uint32_t tmem_p, int h,
                                                 uint32_t vd, uint32_t idesc, bool first) {
    constexpr int STEPS = T::VROW_KEYS / 16;
#pragma unroll
    for (int kk = 0; kk < STEPS; ++kk)
        umma_ts_lo(tmem_o, tmem_p + (h * STEPS + kk) * 8, vd + (uint32_t)((kk * 2048) >> 4), idesc,
                   (!first || h > 0 || kk > 0) ? 1u : 0u);
}

// MMA issue: one elected lane of one warp issues every tcgen05.mma of the CTA
// and the commits that release K/V slots and signal the softmax/correction
// warpgroups.
template <class T, bool VARLEN>
__device__ void prefill_mma_role(int tq, const PrefillArgs& a, const PrefillWork& w,
                                 PrefillAux<T>* aux, uint32_t tmem, uint32_t sQ, uint32_t sRing,
                                 const WaitCtx& wc, unsigned long long* tr) {
    // The whole role runs on lane 0: tcgen05.mma and tcgen05.commit are
    // issued by a single thread, and lane-level waits avoid warp collectives
    // on the issue path.  Lanes 1..31 wait at the final __syncwarp.
    const int lane = threadIdx.x & 31;
    const bool leader = true;
    if (lane != 0) {
        __syncwarp();
        return;
    }
    if (tq != 0) tr = nullptr;
    auto full_bar = [&](int p) { return smem_u32(&aux->bar_full[ring_slot<T>(p)]); };
    auto empty_bar = [&](int p) { return smem_u32(&aux->bar_empty[ring_slot<T>(p)]); };
    auto wait_tile = [&](int p0, unsigned site) {
        for (int pc = 0; pc < T::PIECES; ++pc)
            if (!mbar_wait_lane(full_bar(p0 + pc), ring_phase<T>(p0 + pc), wc, kErrWaitTimeout | site))
                return false;
        return true;
    };
    // release a K or V tile once the MMAs issued so far (which read it) complete
    auto release_tile = [&](int p0, bool) {
        if (leader)
            for (int pc = 0; pc < T::PIECES; ++pc) tc_commit(empty_bar(p0 + pc));
    };
    // descriptors of the Q tiles and of ring slot 0, built once; everything
    // else is an address offset added to them
    const uint32_t qd0 = sdesc_lo_sw128(sQ, 16);             // K-major Q
    const uint32_t kd0 = sdesc_lo_sw128(sRing, 16);          // K-major K
    const uint32_t vd0 = sdesc_lo_sw128(sRing, T::CHUNK);    // MN-major V
    auto qdesc = [&](int t) { return qd0 + (uint32_t)((t * T::QTILE) >> 4); };
    auto slot_off = [&](int p) { return (uint32_t)((ring_slot<T>(p) * T::SLOT) >> 4); };
    auto kdesc = [&](int p0, uint32_t (&kd)[T::PIECES]) {
#pragma unroll
        for (int pc = 0; pc < T::PIECES; ++pc) kd[pc] = kd0 + slot_off(p0 + pc);
    };
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t idesc_v = idesc_bf16_f32(128, T::PV_N, false, true);
    uint32_t kd[T::PIECES];

    if (w.n_max > 0) do {
        if (!mbar_wait_lane(smem_u32(&aux->bar_q), 0, wc, kErrWaitTimeout | kSiteMmaQ)) break;
        if constexpr (T::NQ == 2) {
            // one issuing warp alternates the tiles: PV_0(j), S_0(j+1),
            // PV_1(j), S_1(j+1); each softmax overlaps the other tile's MMAs
            if (!wait_tile(0, kSiteMmaK)) break;
            tc_fence_after();
            kdesc(0, kd);
            if (leader) {
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (w.n_kv[t] <= 0) continue;
                    issue_score<T>(tmem + T::s_col(t), qdesc(t), kd, idesc_s);
                    tc_commit(smem_u32(&aux->bar_s_full[t]));
                }
            }
            release_tile(0, false);
            bool ok = true;
            for (int j = 0; j < w.n_max && ok; ++j) {
                const int posV = (2 * j + 1) * T::PIECES;
                const int posK = (2 * j + 2) * T::PIECES;
                const uint32_t ph = (uint32_t)(j & 1);
                if (!wait_tile(posV, kSiteMmaV)) break;
                trace_mark(tr, kTrMma, j, 0);
                bool k_next_ready = false;
#pragma unroll
                for (int t = 0; t < 2; ++t) {
                    if (j >= w.n_kv[t]) continue;
                    if (!mbar_wait_lane(smem_u32(&aux->bar_p_ready[sig_idx<T>(t, j)]),
                                        sig_par<T>(j), wc,
                                   kErrWaitTimeout | kSiteMmaP)) {
                        ok = false;
                        break;
                    }
                    trace_mark(tr, kTrMma, j, 1 + 3 * t);
                    tc_fence_after();
                    if constexpr (T::SEP_P) {
                        // S_t(j+1) first (the softmax has read S_t(j)), then
                        // PV_t(j) from the tile's own P columns
                        if (j + 1 < w.n_kv[t]) {
                            if (!k_next_ready) {
                                if (!wait_tile(posK, kSiteMmaK)) { ok = false; break; }
                                k_next_ready = true;
                                trace_mark(tr, kTrMma, j, 7);
                                kdesc(posK, kd);
                            }
                            tc_fence_after();
                            issue_score<T>(tmem + T::s_col(t), qdesc(t), kd, idesc_s);
                            tc_commit(smem_u32(&aux->bar_s_full[t]));
                            trace_mark(tr, kTrMma, j, 9 + t);
                        }
                    }
                    if (leader) {
                        issue_value<T>(tmem + T::o_col(t), tmem + T::p_col(t),
                                       vd0 + slot_off(posV), idesc_v, j == 0);
                        tc_commit(smem_u32(&aux->bar_pv_done[t]));
                    }
                    // V_j fully consumed after the last tile that uses it (tile 1,
                    // or tile 0 alone when tile 1 has no block j: a packed
                    // sequence may end inside tile 0)
                    if (t == 1 || (VARLEN && j >= w.n_kv[1])) release_tile(posV, false);
                    trace_mark(tr, kTrMma, j, 2 + 3 * t);
                    if (!T::SEP_P && j + 1 < w.n_kv[t]) {
                        if (!k_next_ready) {
                            if (!wait_tile(posK, kSiteMmaK)) { ok = false; break; }
                            k_next_ready = true;
                            trace_mark(tr, kTrMma, j, 7);
                            kdesc(posK, kd);
                        }
                        // S_t(j+1) overwrites P_t(j): PV_t(j) must have completed
                        if (!mbar_wait_lane(smem_u32(&aux->bar_pv_done[t]), ph, wc,
                                       kErrWaitTimeout | kSiteMmaPv)) {
                            ok = false;
                            break;
                        }
                        trace_mark(tr, kTrMma, j, 3 + 3 * t);
                        tc_fence_after();
                        if (leader) {
                            issue_score<T>(tmem + T::s_col(t), qdesc(t), kd, idesc_s);
                            tc_commit(smem_u32(&aux->bar_s_full[t]));
                        }
                        trace_mark(tr, kTrMma, j, 9 + t);
                    }
                }
                if (ok && j + 1 < w.n_max) release_tile(posK, false);
                trace_mark(tr, kTrMma, j, 8);
            }
        } else {
            if (!wait_tile(0, kSiteMmaK)) break;
            tc_fence_after();
            kdesc(0, kd);
            if (leader) {
                issue_score<T>(tmem + T::s_col(0), qdesc(0), kd, idesc_s);
                tc_commit(smem_u32(&aux->bar_s_full[0]));
            }
            release_tile(0, false);
            for (int j = 0; j < w.n_max; ++j) {
                const int posV = (2 * j + 1) * T::PIECES;
                const int posK = (2 * j + 2) * T::PIECES;
                // next score first, into the other buffer; that buffer held
                // P(j-1), so PV(j-1) must have completed
                if (j + 1 < w.n_max) {
                    if (!wait_tile(posK, kSiteMmaK)) break;
                    if (j >= 1 && !mbar_wait_lane(smem_u32(&aux->bar_pv_done[sig_idx<T>(0, j - 1)]),
                                                  sig_par<T>(j - 1), wc,
                                                  kErrWaitTimeout | kSiteMmaPv))
                        break;
                    tc_fence_after();
                    kdesc(posK, kd);
                    if (leader) {
                        issue_score<T>(tmem + T::s_col((j + 1) & 1), qdesc(0), kd, idesc_s);
                        tc_commit(smem_u32(&aux->bar_s_full[(j + 1) & 1]));
                    }
                    release_tile(posK, false);
                }
                if (!wait_tile(posV, kSiteMmaV)) break;
                trace_mark(tr, kTrMma, j, 0);
                if (!mbar_wait_lane(smem_u32(&aux->bar_p_ready[sig_idx<T>(0, j)]), sig_par<T>(j), wc,
                               kErrWaitTimeout | kSiteMmaP))
                    break;
                trace_mark(tr, kTrMma, j, 1);
                tc_fence_after();
                if (leader) {
#pragma unroll
                    for (int nh = 0; nh < T::PIECES; ++nh)
                        issue_value<T>(tmem + T::o_col(0) + nh * 128,
                                       tmem + T::s_col(j & 1) + 64, vd0 + slot_off(posV + nh),
                                       idesc_v, j == 0);
                    tc_commit(smem_u32(&aux->bar_pv_done[sig_idx<T>(0, j)]));
                }
                release_tile(posV, false);
                trace_mark(tr, kTrMma, j, 2);
            }
        }
    } while (0);
    // All MMAs issued by this warp must have completed before tensor memory
    // is freed.
    {
        const uint32_t drain = smem_u32(&aux->bar_drain[tq]);
        tc_commit(drain);
        mbar_wait_drain(drain, 0, a.wait_limit_ns);
    }
    __syncwarp();
}

// ------------------------------------ split output columns (head_dim 512) ----
//
// With DV_SPLIT > 1 a CTA holds the whole 128 x 512 Q tile (128 KB) and
// streams K and its own 256 columns of V through five one-chunk (16 KB) ring
// slots.  The ring is filled in the order the MMA warp consumes it -- K_0,
// then K_{j+1} before V_j -- because with one Q tile the score MMA of block
// j+1 is issued before the value MMA of block j, and five slots cannot hold
// a value tile while a whole key tile waits behind it.  Each K piece is
// released as soon as its four K-steps have been issued and completed.

// Loads ring position p (then p + 1): the 64-column chunks
// [pc SLOT_CH, (pc + 1) SLOT_CH) of K_j (is_v false) or of the CTA's part of
// V_j.  A partial last value tile is zeroed past the sequence end before it
// is published; `ntail` counts those copies (the parity of bar_tail).
// Executed by the producer warp (lane 0 issues).
template <class T, bool VARLEN>
__device__ __forceinline__ bool load_piece(const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                           const PrefillArgs& a, const PrefillWork& w,
                                           PrefillAux<T>* aux, uint32_t sRing, const WaitCtx& wc,
                                           unsigned long long* tr, int j, bool is_v, int pc,
                                           int& p, int& ntail) {
    const int lane = threadIdx.x & 31;
    const uint32_t slot = ring_slot<T>(p);
    if (!mbar_wait(smem_u32(&aux->bar_empty[slot]), ring_phase<T>(p) ^ 1u, wc,
                   kErrWaitTimeout | kSiteLoadEmpty))
        return false;
    trace_mark(tr, kTrLoad, p >> 4, p & 15);   // position p's copy issued
    const uint32_t full = smem_u32(&aux->bar_full[slot]);
    const uint32_t dst = sRing + slot * T::SLOT;
    const int jk = w.kb + j;
    const int rv = w.L - jk * T::BN;
    int ty = (VARLEN ? w.k0 : 0) + jk * T::BN, tz = VARLEN ? w.hk : w.b * a.Hkv + w.hk;
    if (a.block_table != nullptr) {
        const int page = a.block_table[(size_t)w.b * a.max_pages + ty / a.page_size];
        ty = ty % a.page_size;
        tz = page * a.Hkv + w.hk;
    }
    if (T::VROWS && is_v) {
        // keys [VROW_KEYS pc, +VROW_KEYS) of V_j, the CTA's 256 columns (one
        // 4-D copy of four chunks); rows past the sequence end zeroed
        constexpr int RK = T::VROW_KEYS;
        const int r0 = rv - RK * pc;
        const uint32_t bar = (r0 < RK) ? smem_u32(&aux->bar_tail) : full;
        if (lane == 0) {
            mbar_arrive_expect_tx(bar, (uint32_t)T::SLOT);
            tma_load_4d(dst, tm_v, 0, ty + RK * pc, w.dv0 / 64, tz, bar);
        }
        if (r0 < RK) {
            if (!mbar_wait(bar, (uint32_t)(ntail & 1), wc, kErrWaitTimeout | kSiteLoadTail))
                return false;
            ++ntail;
            zero_value_rows<T>(dst, r0 > 0 ? r0 : 0);
            if (lane == 0) mbar_arrive(full);
        }
        __syncwarp();
        ++p;
        return true;
    }
    const int c0 = pc * T::SLOT_CH + (is_v ? w.dv0 / 64 : 0);   // first chunk of the slot
    if (is_v && j == w.n_max - 1 && rv < T::BN) {
        // partial last value tile: rows [rv, BN) zeroed before publication
        const uint32_t tail = smem_u32(&aux->bar_tail);
        if (lane == 0) {
            mbar_arrive_expect_tx(tail, (uint32_t)T::SLOT);
            load_chunks<T, T::SLOT_CH>(dst, tm_v, c0, ty, tz, tail);
        }
        if (!mbar_wait(tail, (uint32_t)(ntail & 1), wc, kErrWaitTimeout | kSiteLoadTail))
            return false;
        ++ntail;
        zero_value_tail<T>(dst, rv);
        if (lane == 0) mbar_arrive(full);
    } else if (lane == 0) {
        mbar_arrive_expect_tx(full, (uint32_t)T::SLOT);
        load_chunks<T, T::SLOT_CH>(dst, is_v ? tm_v : tm_k, c0, ty, tz, full);
    }
    __syncwarp();
    ++p;
    return true;
}

// Producer: Q once, then the pieces in consumption order.
template <class T, bool CAUSAL, bool WINDOW, bool VARLEN>
__device__ void prefill_load_role_dv(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                     const CUtensorMap* tm_v, const PrefillArgs& a,
                                     const PrefillWork& w, PrefillAux<T>* aux, uint32_t sQ,
                                     uint32_t sRing, const WaitCtx& wc, unsigned long long* tr) {
    const int lane = threadIdx.x & 31;
    if (lane != 0) tr = nullptr;
    if (w.n_max <= 0) return;
    const uint32_t bar_q = smem_u32(&aux->bar_q);
    if (lane == 0) {
        tma_prefetch_desc(tm_q);
        tma_prefetch_desc(tm_k);
        tma_prefetch_desc(tm_v);
        mbar_arrive_expect_tx(bar_q, (uint32_t)T::QTILE);
        load_chunks<T, T::NCH>(sQ, tm_q, 0, (VARLEN ? w.q0 : 0) + w.row0,
                               VARLEN ? w.h : w.b * a.Hq + w.h, bar_q);
    }
    int p = 0;       // ring position of the next piece
    int ntail = 0;   // partial value pieces loaded so far
    auto load = [&](int j, bool is_v, int pc) -> bool {
        return load_piece<T, VARLEN>(tm_k, tm_v, a, w, aux, sRing, wc, tr, j, is_v, pc, p, ntail);
    };
    bool ok = true;
    for (int pc = 0; pc < T::PIECES && ok; ++pc) ok = load(0, false, pc);
    if (ok && lane == 0 && a.q_prefetch > 0 &&
        (int)blockIdx.x + a.q_prefetch * T::DV_SPLIT < (int)gridDim.x)
        prefetch_q_of<T, CAUSAL, WINDOW, VARLEN>(tm_q, a,
                                                 (int)blockIdx.x + a.q_prefetch * T::DV_SPLIT);
    for (int j = 0; j < w.n_max && ok; ++j) {
        if (j + 1 < w.n_max)
            for (int pc = 0; pc < T::PIECES && ok; ++pc) ok = load(j + 1, false, pc);
        for (int pc = 0; pc < T::VPIECES && ok; ++pc) ok = load(j, true, pc);
    }
    // every copy issued must have landed before the CTA exits
    if (lane == 0) {
        mbar_wait_drain(bar_q, 0, a.wait_limit_ns);
        for (int q = p > T::NSLOT ? p - T::NSLOT : 0; q < p; ++q)
            mbar_wait_drain(smem_u32(&aux->bar_full[ring_slot<T>(q)]), ring_phase<T>(q),
                            a.wait_limit_ns);
    }
    __syncwarp();
}

// MMA issue (one lane): S(0); then per block j: S(j+1) into the other score
// buffer (once PV(j-1), which read that buffer's P, has completed), and
// PV(j) over the CTA's output columns, one N = 64 chunk per ring piece.
template <class T>
__device__ void prefill_mma_role_dv(const PrefillArgs& a, const PrefillWork& w,
                                    PrefillAux<T>* aux, uint32_t tmem, uint32_t sQ,
                                    uint32_t sRing, const WaitCtx& wc, unsigned long long* tr) {
    const int lane = threadIdx.x & 31;
    if (lane != 0) {
        __syncwarp();
        return;
    }
    const uint32_t qd0 = sdesc_lo_sw128(sQ, 16);
    const uint32_t kd0 = sdesc_lo_sw128(sRing, 16);
    const uint32_t vd0 = sdesc_lo_sw128(sRing, T::CHUNK);
    const uint32_t vd0r = sdesc_lo_sw128(sRing, T::VROW_CHUNK);   // row-split V slots
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t idesc_v = idesc_bf16_f32(128, T::PV_N, false, true);
    int p = 0;   // ring position of the next piece (the producer's order)
    auto next_piece = [&](unsigned site) -> bool {
        if (!mbar_wait_lane(smem_u32(&aux->bar_full[ring_slot<T>(p)]), ring_phase<T>(p), wc,
                            kErrWaitTimeout | site))
            return false;
        tc_fence_after();
        return true;
    };
    auto slot_desc = [&](uint32_t d0) { return d0 + (uint32_t)((ring_slot<T>(p) * T::SLOT) >> 4); };
    // S(buffer sb) = Q K^T, each K piece released once its K-steps complete
    // (trace: row j = the block whose scores these are, events 1..8 = pieces)
    auto score = [&](int sb, int jt) -> bool {
        for (int pc = 0; pc < T::PIECES; ++pc) {
            if (!next_piece(kSiteMmaK)) return false;
            trace_mark(tr, kTrMma, jt, 1 + pc);
            const uint32_t kd = slot_desc(kd0);
#pragma unroll
            for (int kin = 0; kin < T::SLOT_CH * 4; ++kin) {
                const int kk = pc * T::SLOT_CH * 4 + kin;
                umma_ss_lo(tmem + T::s_col(sb), qd0 + kstep_off(kk), kd + kstep_off(kin), idesc_s,
                           kk > 0 ? 1u : 0u);
            }
            tc_commit(smem_u32(&aux->bar_empty[ring_slot<T>(p)]));
            ++p;
        }
        tc_commit(smem_u32(&aux->bar_s_full[sb]));
        return true;
    };
    if (w.n_max > 0) do {
        if (!mbar_wait_lane(smem_u32(&aux->bar_q), 0, wc, kErrWaitTimeout | kSiteMmaQ)) break;
        tc_fence_after();
        if (!score(0, 0)) break;
        bool ok = true;
        for (int j = 0; j < w.n_max && ok; ++j) {
            if (j + 1 < w.n_max) {
                if (j >= 1 && !mbar_wait_lane(smem_u32(&aux->bar_pv_done[sig_idx<T>(0, j - 1)]),
                                              sig_par<T>(j - 1), wc, kErrWaitTimeout | kSiteMmaPv))
                    break;
                tc_fence_after();
                trace_mark(tr, kTrMma, j + 1, 0);   // S(j+1) may start
                if (!score((j + 1) & 1, j + 1)) break;
            }
            if (!mbar_wait_lane(smem_u32(&aux->bar_p_ready[sig_idx<T>(0, j)]), sig_par<T>(j), wc,
                                kErrWaitTimeout | kSiteMmaP))
                break;
            trace_mark(tr, kTrMma, j, 9);             // P(j) ready
            tc_fence_after();
            for (int nh = 0; nh < T::VPIECES; ++nh) {
                if (!next_piece(kSiteMmaV)) {
                    ok = false;
                    break;
                }
                trace_mark(tr, kTrMma, j, 10 + nh);   // V piece nh landed
                if constexpr (T::VROWS)
                    issue_value_rows<T>(tmem + T::o_col(0), tmem + T::s_col(j & 1) + 64, nh,
                                        slot_desc(vd0r), idesc_v, j == 0);
                else
                    issue_value<T>(tmem + T::o_col(0) + nh * T::PV_N, tmem + T::s_col(j & 1) + 64,
                                   slot_desc(vd0), idesc_v, j == 0);
                tc_commit(smem_u32(&aux->bar_empty[ring_slot<T>(p)]));
                ++p;
            }
            if (ok) tc_commit(smem_u32(&aux->bar_pv_done[sig_idx<T>(0, j)]));
        }
    } while (0);
    {
        const uint32_t drain = smem_u32(&aux->bar_drain[0]);
        tc_commit(drain);
        mbar_wait_drain(drain, 0, a.wait_limit_ns);
    }
    __syncwarp();
}

// Stages 32-column groups [c_begin, c_end) of one Q tile's O row r as bf16
// (O * inv_l) into the 128-byte-swizzled staging tile at `stage` (nk == 0:
// zeros).  Called by one warpgroup (thread = row = tensor-memory lane).
template <class T>
__device__ __forceinline__ void stage_o_rows(uint32_t lane_base, uint32_t o_col, uint32_t stage,
                                             int r, int nk, float inv_l, int c_begin, int c_end) {
#pragma unroll 1
    for (int c32 = c_begin; c32 < c_end; ++c32) {
        uint32_t v[32];
        if (nk > 0) {
            tmem_ld32(lane_base + o_col + c32 * 32, v);
            tmem_wait_ld();
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0u;
        }
        const uint32_t row_addr = stage + (c32 >> 1) * T::CHUNK + r * 128;
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) {
            const int g = (c32 & 1) * 4 + g4;    // 16-byte granule within the 128-byte row
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                pk[e] = pack_bf16x2(__uint_as_float(v[g4 * 8 + 2 * e]) * inv_l,
                                    __uint_as_float(v[g4 * 8 + 2 * e + 1]) * inv_l);
            const uint32_t addr = row_addr + ((uint32_t)(g ^ (r & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[0]),
                         "r"(pk[1]), "r"(pk[2]), "r"(pk[3])
                         : "memory");
        }
    }
}

// Writes 32-column groups [c_begin, c_end) of one O row (O * inv_l, bf16)
// straight to global memory at orow (nk == 0: zeros); rows past the query
// length write nothing.
template <class T>
__device__ __forceinline__ void store_o_rows_direct(uint32_t lane_base, uint32_t o_col,
                                                    uint16_t* orow, bool row_ok, int nk,
                                                    float inv_l, int c_begin, int c_end) {
#pragma unroll 1
    for (int c32 = c_begin; c32 < c_end; ++c32) {
        uint32_t v[32];
        if (nk > 0) {
            tmem_ld32(lane_base + o_col + c32 * 32, v);
            tmem_wait_ld();
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0u;
        }
        if (!row_ok) continue;
#pragma unroll
        for (int g4 = 0; g4 < 4; ++g4) {
            uint32_t pk[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                pk[e] = pack_bf16x2(__uint_as_float(v[g4 * 8 + 2 * e]) * inv_l,
                                    __uint_as_float(v[g4 * 8 + 2 * e + 1]) * inv_l);
            *reinterpret_cast<uint4*>(orow + c32 * 32 + g4 * 8) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
    }
}

// The O staging buffers (STAGE_BUFS x 2 KB) of warp `warp` of a warpgroup
// (its index within the group), after the barrier block.
template <class T>
__device__ __forceinline__ uint32_t stage_of(uint32_t sQ, int warp) {
    return sQ + T::SMEM_Q + T::SMEM_RING + T::SMEM_AUX +
           (uint32_t)(warp & 3) * (uint32_t)(T::STAGE_BUFS * 2048);
}

// Writes 32-column groups [c_begin, c_end) of the calling warp's 32 O rows
// (O * inv_l, bf16; nk == 0: zeros) through the warp's 2 KB staging area at
// `stage`.  NG groups are read from tensor memory per wait (the load latency
// dominates otherwise); then, group by group, each lane writes its row's 64
// bytes (16-byte chunks XOR-swizzled by row pair, 4-way bank conflicts at
// most) and each store instruction writes 8 rows x 64 contiguous bytes (4
// lanes per row) instead of 32 scattered 16-byte pieces.  obase: the warp's
// first row at its first column; rows past nvalid are not written.
//
// With a 32 x 32 O map (tm_o32 non-null: box {32 columns, 32 rows, 1}, 64-byte
// swizzle, whose layout is exactly this staging layout) one lane stores each
// group with a TMA store instead, at (ox + 32 c, oy, oz), rotating over
// STAGE_BUFS staging buffers: a buffer is rewritten once the store that last
// used it has read it.
template <class T, int NG>
__device__ __forceinline__ void store_o_rows_staged(uint32_t lane_base, uint32_t o_col,
                                                    uint16_t* obase, size_t row_stride,
                                                    int nvalid, int nk, float inv_l,
                                                    int c_begin, int c_end, uint32_t stage,
                                                    const CUtensorMap* tm_o32 = nullptr,
                                                    int ox = 0, int oy = 0, int oz = 0) {
    const int lane = threadIdx.x & 31;
    constexpr int NB = T::STAGE_BUFS > 0 ? T::STAGE_BUFS : 1;
    int nst = 0;   // TMA stores issued by this call
    if (tm_o32 != nullptr) {   // an earlier call's stores must have read the buffers
        if (lane == 0) bulk_wait_group_read_0();
        __syncwarp();
    }
#pragma unroll 1
    for (int cb = c_begin; cb < c_end; cb += NG) {
        uint32_t v[NG][32];
        if (nk > 0) {
#pragma unroll
            for (int g = 0; g < NG; ++g)
                if (cb + g < c_end) tmem_ld32(lane_base + o_col + (cb + g) * 32, v[g]);
            tmem_wait_ld();
        } else {
#pragma unroll
            for (int g = 0; g < NG; ++g)
#pragma unroll
                for (int e = 0; e < 32; ++e) v[g][e] = 0u;
        }
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            const int c32 = cb + g;
            if (c32 >= c_end) break;
            const uint32_t buf = (tm_o32 != nullptr) ? stage + (uint32_t)(nst % NB) * 2048u : stage;
            if (tm_o32 != nullptr && nst >= NB) {   // the store that last used buf has read it
                if (lane == 0) bulk_wait_group_read<NB - 1>();
                __syncwarp();
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    pk[e] = pack_bf16x2(__uint_as_float(v[g][i * 8 + 2 * e]) * inv_l,
                                        __uint_as_float(v[g][i * 8 + 2 * e + 1]) * inv_l);
                const uint32_t dst = buf + lane * 64 + ((i ^ ((lane >> 1) & 3)) << 4);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(pk[0]),
                             "r"(pk[1]), "r"(pk[2]), "r"(pk[3])
                             : "memory");
            }
            if (tm_o32 != nullptr) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_3d(tm_o32, buf, ox + c32 * 32, oy, oz);
                    bulk_commit_group();
                }
                ++nst;
                continue;
            }
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int rr = 8 * k + (lane >> 2), c = lane & 3;
                uint32_t x0, x1, x2, x3;
                asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                             : "=r"(x0), "=r"(x1), "=r"(x2), "=r"(x3)
                             : "r"(stage + rr * 64 + ((c ^ ((rr >> 1) & 3)) << 4))
                             : "memory");
                if (rr < nvalid)
                    *reinterpret_cast<uint4*>(obase + (size_t)rr * row_stride + c32 * 32 + c * 8) =
                        make_uint4(x0, x1, x2, x3);
            }
            __syncwarp();
        }
    }
}

// Final normaliser of a row: the row sum l and max m (log2 units) of its
// visible keys, plus the head's attention sink (one more term e^{sigma}
// without a value, O rebased to max(m, sigma)).  Returns 1 / l' scaled by
// that rebase, and sets lf / mf to the final sum and max.
__device__ __forceinline__ float final_scale(const PrefillArgs& a, int h, float l, float m,
                                             float& lf, float& mf) {
    lf = l;
    mf = m;
    float oscale = 1.f;
    if (a.sinks != nullptr) {
        const float sg = a.sinks[h] * kLog2e;
        const float m2 = fmaxf(m, sg);
        if (m2 == -INFINITY) {
            lf = 0.f;
        } else {
            oscale = (m == -INFINITY) ? 0.f : ex2_approx(m - m2);
            lf = l * oscale + ex2_approx(sg - m2);
            mf = m2;
        }
    }
    return (lf > 0.f) ? oscale / lf : 0.f;
}

// Whether a kernel splits its epilogue between the softmax and correction
// warpgroups: the one-tile kernels (head_dim 256, 512) and the masked
// (causal or windowed) two-tile ones, where it measured 1-2 % faster on
// GB300; in the unmasked two-tile kernels it measured ~1 % slower (their
// softmax runs closer to its register budget).  Packed sequences store
// row by row from the correction warpgroup.
template <class T, bool MASKED, bool VARLEN>
__host__ __device__ constexpr bool epi_split() {
    return T::EPI_SPLIT > 0 && !VARLEN && (T::NQ == 1 || MASKED);
}

// The softmax warpgroup's part of tile t's epilogue (dense launches of
// whole units): O chunks [0, EPI_SPLIT) staged and stored by this
// warpgroup once the last value MMA of the tile has completed.
template <class T, bool VARLEN, bool ENABLED>
__device__ void softmax_epilogue_part(int t, const CUtensorMap* tm_o, const PrefillArgs& a,
                                      const PrefillWork& w, PrefillAux<T>* aux, uint32_t tmem,
                                      uint32_t sQ, float l, float m, const WaitCtx& wc, int J0) {
    if constexpr (!ENABLED) {
        return;
    } else {
        if (w.piece >= 0) return;   // pieces of split units: the correction writes them
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int r = (warp & 3) * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const int nk = w.n_kv[t];
        if (nk > 0) {
            if (!mbar_wait(smem_u32(&aux->bar_pv_done[sig_idx<T>(t, J0 + nk - 1)]),
                           sig_par<T>(J0 + nk - 1), wc, kErrWaitTimeout | kSiteEpiPv))
                return;
            tc_fence_after();
        }
        float lf, mf;
        const float inv_l = final_scale(a, w.h, l, m, lf, mf);
        const uint32_t stage = sQ + t * T::QTILE;
        stage_o_rows<T>(lane_base, T::o_col(t), stage, r, nk, inv_l, 0, 2 * T::EPI_SPLIT);
        fence_proxy_async_smem();
        mbar_arrive_warp(smem_u32(&aux->bar_epi_sm[t]));
        if ((warp & 3) == 0 && lane == 0 && w.row0 + t * T::BM < a.Sq &&
            mbar_wait_lane(smem_u32(&aux->bar_epi_sm[t]), 0, wc, kErrWaitTimeout | kSiteEpiStage)) {
#pragma unroll
            for (int ch = 0; ch < T::EPI_SPLIT; ++ch)
                tma_store_3d(tm_o, stage + ch * T::CHUNK, w.dv0 + ch * 64, w.row0 + t * T::BM,
                             w.b * a.Hq + w.h);
            bulk_commit_group();
            bulk_wait_group_read_0();   // the CTA may exit once shared memory was read
        }
    }
}

// ------------------------------------------------------------- softmax ----

// PERSIST (one Q tile, persistent kernel): the unit is one of several that
// this CTA processes; J0 counts the key blocks of its earlier units, and the
// barriers, mailboxes and score buffers are indexed by the CTA-wide block
// index J0 + j.
template <class T, bool CAUSAL, bool WINDOW, bool VARLEN, bool PERSIST = false>
__device__ void prefill_softmax_role(int t, const CUtensorMap* tm_o, const PrefillArgs& a,
                                     const PrefillWork& w, PrefillAux<T>* aux, uint32_t tmem,
                                     uint32_t sQ, const WaitCtx& wc, unsigned long long* tr,
                                     int J0 = 0, int kq = 0) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if ((warp & 3) != 0 || lane != 0) tr = nullptr;
    const int trole = t == 0 ? kTrSoftmax0 : kTrSoftmax1;
    const int r = (warp & 3) * 32 + lane;                    // tile row = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const int row = w.row0 + t * T::BM + r;
    int lim = w.L - 1;                                       // last visible key of this row
    if (CAUSAL) lim = min(lim, row + w.off);
    lim -= w.kb * T::BN;   // keys counted from the piece's first key block
    // first visible key of this row (sliding window), same origin; the
    // kernels without a window compile none of this
    const int lo = WINDOW ? row + w.off - a.window + 1 - w.kb * T::BN : 0;
    const float sl2 = a.scale_log2;
    const int nk = w.n_kv[t];
    float m_run = -INFINITY;   // running max of scaled scores, log2 units (the basis)
    float l_run = 0.f;         // running row_sum in that basis
    bool ok = true;
    for (int j = 0; j < nk; ++j) {
        const int J = J0 + j;   // block index over the CTA's units
        const int sb = (T::NSBUF == 2) ? (J & 1) : 0;
        const uint32_t scol = (T::NQ == 2) ? T::s_col(t) : T::s_col(sb);
        uint32_t u[4][32];
        {
            const uint32_t bar_s = smem_u32(&aux->bar_s_full[(T::NQ == 2) ? t : sb]);
            const uint32_t par_s = (T::NQ == 2) ? (uint32_t)(j & 1) : (uint32_t)((J >> 1) & 1);
            if (!mbar_wait(bar_s, par_s, wc, kErrWaitTimeout | kSiteSmS)) {
                ok = false;
                break;
            }
            trace_mark(tr, trole, J, 0);
            trace_mark(tr, trole, J, 1);
            tc_fence_after();
            // two 64-column loads (measured +1 % at head_dim 64 and on the
            // non-causal head_dim-256 shape against four 32-column ones)
            tmem_ld64(lane_base + scol, *reinterpret_cast<uint32_t(*)[2][32]>(&u[0][0]));
            tmem_ld64(lane_base + scol + 64, *reinterpret_cast<uint32_t(*)[2][32]>(&u[2][0]));
        }
        tmem_wait_ld();
        trace_mark(tr, trole, J, 2);
        float s[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(u[c >> 5][c & 31]);
        // mask: only tiles that reach past this row's last visible key
        const int kv0 = j * T::BN;   // relative to the piece's first key (lim is too)
        const bool masked = lim - kv0 < T::BN - 1 || (WINDOW && lo - kv0 > 0);
        const bool warp_masked = __any_sync(0xffffffffu, masked);
        if (masked) {
            const int nvis = lim - kv0 + 1;                  // visible columns [c0, nvis)
            const int c0 = WINDOW ? lo - kv0 : 0;
#pragma unroll
            for (int c = 0; c < 128; ++c)
                s[c] = (c < nvis && (!WINDOW || c >= c0)) ? s[c] : -INFINITY;
        }
        // row max: four independent 3-input-max chains, then combine
        float mq[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float m = fmax3(s[32 * q], s[32 * q + 1], s[32 * q + 2]);
#pragma unroll
            for (int c = 3; c < 31; c += 2) m = fmax3(m, s[32 * q + c], s[32 * q + c + 1]);
            mq[q] = fmaxf(m, s[32 * q + 31]);
        }
        const float mx = fmaxf(fmax3(mq[0], mq[1], mq[2]), mq[3]);
        const float m_new = fmaxf(m_run, mx * sl2);
        float alpha = 1.f;
        if (m_new > m_run + kRescaleThreshold) {
            alpha = ex2_approx(m_run - m_new);   // 0 when m_run = -inf
            m_run = m_new;
        }
        // Mailbox message j: the rebase factor, for the correction warpgroup.
        // The slot is free without a handshake: S(j) was issued after the
        // value MMA of the last block that used the same slot (j-1 for
        // NQ = 2, j-2 for NQ = 1), which waited for the correction's arrive
        // on P-ready, made after it had read that block's message.
        aux->mb_alpha[sig_idx<T>(t, J)][r] = alpha;
        mbar_arrive_warp(smem_u32(&aux->bar_mb_full[sig_idx<T>(t, J)]));
        trace_mark(tr, trole, J, 3);
        // P(j) columns: the upper half of the score buffer, or (SEP_P) the
        // tile's own P columns, which PV_t(j-1) may still be reading
        const uint32_t pcol = T::SEP_P ? T::p_col(t) : scol + 64;
        if (T::SEP_P && j > 0) {
            if (!mbar_wait(smem_u32(&aux->bar_pv_done[sig_idx<T>(t, J - 1)]), sig_par<T>(J - 1), wc,
                           kErrWaitTimeout | kSiteSmPv)) {
                ok = false;
                break;
            }
            tc_fence_after();
        }
        const float base = (m_run == -INFINITY) ? 0.f : m_run;
        const float2 sl2x2 = make_float2(sl2, sl2);
        const float2 nbase = make_float2(-base, -base);
        float2 rs[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                        make_float2(0.f, 0.f)};
        uint32_t pk[2][32];
        if (kUsePolyExp2 && warp_masked) {
            // masked entries are -inf and must give exactly 0: hardware ex2
            // only (without the polynomial option both loops are the same,
            // and only the one below is compiled)
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                const float2 x = ffma2(make_float2(s[2 * c], s[2 * c + 1]), sl2x2, nbase);
                const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
                rs[c & 3] = fadd2(rs[c & 3], p);
                pk[c >> 5][c & 31] = pack_bf16x2(p.x, p.y);
            }
        } else {
#pragma unroll
            for (int c = 0; c < 64; ++c) {
                const float2 x = ffma2(make_float2(s[2 * c], s[2 * c + 1]), sl2x2, nbase);
                const float2 p = (kUsePolyExp2 && c % kPolyEvery == kPolyEvery - 1)
                                     ? exp2_poly_x2(x)
                                     : make_float2(ex2_approx(x.x), ex2_approx(x.y));
                rs[c & 3] = fadd2(rs[c & 3], p);
                pk[c >> 5][c & 31] = pack_bf16x2(p.x, p.y);
                // keys 0..63 go to columns 64..95, whose scores are already in
                // registers: store them early to shorten the live range
                if (c == 31) tmem_st32(lane_base + pcol, pk[0]);
            }
        }
        const float2 rs01 = fadd2(rs[0], rs[1]), rs23 = fadd2(rs[2], rs[3]);
        const float2 rsum = fadd2(rs01, rs23);
        l_run = fmaf(l_run, alpha, rsum.x + rsum.y);
        trace_mark(tr, trole, J, 4);
        if (kUsePolyExp2 && warp_masked) tmem_st32(lane_base + pcol, pk[0]);
        tmem_st32(lane_base + pcol + 32, pk[1]);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive_warp(smem_u32(&aux->bar_p_ready[sig_idx<T>(t, J)]));
        trace_mark(tr, trole, J, 5);
    }
    // persistent kernel: the previous unit's statistics must have been read
    // (the correction warpgroup arrives on O-drained after reading them)
    if (PERSIST && ok && kq > 0)
        ok = mbar_wait(smem_u32(&aux->bar_odrained), (uint32_t)((kq - 1) & 1), wc,
                       kErrWaitTimeout | kSiteSmOdrained);
    if (ok) {   // final row statistics for the epilogue (own slots, own barrier)
        aux->mb_l[t][r] = l_run;
        aux->mb_m[t][r] = m_run;
        mbar_arrive_warp(smem_u32(&aux->bar_fin[t]));
        // (the persistent kernel's correction warpgroup drains all of O)
        softmax_epilogue_part<T, VARLEN, epi_split<T, CAUSAL || WINDOW, VARLEN>() && !PERSIST>(
            t, tm_o, a, w, aux, tmem, sQ, l_run, m_run, wc, J0);
    }
}

// ---------------------------------------------------- correction/epilogue ----

// Stores 32 columns of one output row as bf16: O = v * inv_l.
__device__ __forceinline__ void store_o32(uint16_t* orow, const float (&v)[32], float inv_l) {
    uint4* dst = reinterpret_cast<uint4*>(orow);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 x;
        x.x = pack_bf16x2(v[8 * q + 0] * inv_l, v[8 * q + 1] * inv_l);
        x.y = pack_bf16x2(v[8 * q + 2] * inv_l, v[8 * q + 3] * inv_l);
        x.z = pack_bf16x2(v[8 * q + 4] * inv_l, v[8 * q + 5] * inv_l);
        x.w = pack_bf16x2(v[8 * q + 6] * inv_l, v[8 * q + 7] * inv_l);
        dst[q] = x;
    }
}

// Arrival of a piece of a split unit, once its partial result (unnormalised
// O, row max, row sum) is in scratch: the pieces count themselves on the
// unit's counter, and the one that arrives last sets aux->merge_last; its CTA
// then merges the unit at the end of the kernel (merge_unit, all threads).
// No CTA waits for another.
template <class T, class Aux>
__device__ void split_arrive(const PrefillArgs& a, const PrefillWork& w, Aux* aux,
                             const WaitCtx& wc) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    mbar_arrive_warp(smem_u32(&aux->bar_split_a));   // this warp's stores issued
    if (warp != T::CORR_WG * 4) return;
    if (!mbar_wait(smem_u32(&aux->bar_split_a), 0, wc, kErrWaitTimeout | kSiteSplitA) || lane != 0)
        return;
    __threadfence();   // this piece's stores (all four warps) before the count
    unsigned long long* cp = a.part_count + w.tail;
    const unsigned long long tag = a.epoch << 16;
    unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(cp);
    unsigned long long arrived = 0;
    for (int attempt = 0; attempt <= a.split; ++attempt) {
        const unsigned long long cur = ((old >> 16) == a.epoch) ? (old & 0xffffull) : 0ull;
        const unsigned long long prev = atomicCAS(cp, old, tag | (cur + 1));
        if (prev == old) {
            arrived = cur + 1;
            break;
        }
        old = prev;
    }
    if (arrived == 0) record_error(wc, kErrSplitCount);
    // The last piece resets the counter (no other piece touches it again in
    // this launch), so that a replay of a captured launch -- same scratch
    // address, same epoch -- starts from zero.
    if (arrived == (unsigned long long)a.split)
        *reinterpret_cast<volatile unsigned long long*>(cp) = 0ull;
    __threadfence();   // the other pieces' stores before this CTA's loads
    // what the merge needs, kept in shared memory rather than live in
    // registers through every role
    aux->merge_unit[0] = w.tail;
    aux->merge_unit[1] = w.h;
    aux->merge_unit[2] = w.b;
    aux->merge_unit[3] = w.row0;
    aux->merge_last = arrived == (unsigned long long)a.split ? 1 : 0;
}

// Merge of split unit w.tail once all its pieces' partial results are in
// scratch: each piece's O, row max and row sum are rebased to the running
// max and added (the streaming recurrence again, over pieces instead of key
// blocks; the sink, if any, is one more term without a value), then
// O / row_sum and LSE are stored.  The work (rows x 16-column groups, rows
// fastest so that loads coalesce) is dealt to threads tid = 0 .. nthr-1; a
// thread's loads for one piece do not depend on the previous piece, so two
// pieces' loads are in flight at once.
// Unit: split index `tail`, query head h, batch entry b, first row row0.
template <class T>
__device__ void merge_unit(const PrefillArgs& a, int tail, int h, int b, int row0, int tid,
                           int nthr) {
    constexpr int NC16 = T::D_COLS / 16;
    const int s0 = tail * a.split;
    // head-packed tiles (a.pack > 1): row r is head h + r / R at position
    // row0 + r % R, R = BM / pack
    const int prows = T::BM / (a.pack > 1 ? a.pack : 1);
#pragma unroll 1
    for (int task = tid; task < T::NQ * NC16 * T::BM; task += nthr) {
        const int r = task % T::BM;
        const int c16 = (task / T::BM) % NC16;
        const int t = task / (T::BM * NC16);
        const int hr = a.pack > 1 ? h + r / prows : h;
        const int row = a.pack > 1 ? row0 + r % prows : row0 + t * T::BM + r;
        if (row >= a.Sq) continue;
        const float sg = (a.sinks != nullptr) ? a.sinks[hr] * kLog2e : -INFINITY;
        float M = sg;
        float L = (sg == -INFINITY) ? 0.f : 1.f;
        float acc[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[e] = 0.f;
#pragma unroll 2
        for (int k = 0; k < a.split; ++k) {
            const size_t slot = (size_t)(s0 + k) * T::NQ + t;
            const float* ml = a.part_ml + slot * 2 * T::BM;
            const float4* po = reinterpret_cast<const float4*>(a.part_o + slot * (T::D_COLS * T::BM));
            const float mk = __ldcg(ml + r);
            const float lk = __ldcg(ml + T::BM + r);
            float4 x[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) x[q] = __ldcg(po + (size_t)(c16 * 4 + q) * T::BM + r);
            if (mk == -INFINITY) continue;   // a piece without keys adds nothing
            const float m2 = fmaxf(M, mk);
            const float sc = (M == -INFINITY) ? 0.f : ex2_approx(M - m2);
            const float wk = ex2_approx(mk - m2);
            M = m2;
            L = fmaf(L, sc, wk * lk);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc[4 * q + 0] = fmaf(acc[4 * q + 0], sc, wk * x[q].x);
                acc[4 * q + 1] = fmaf(acc[4 * q + 1], sc, wk * x[q].y);
                acc[4 * q + 2] = fmaf(acc[4 * q + 2], sc, wk * x[q].z);
                acc[4 * q + 3] = fmaf(acc[4 * q + 3], sc, wk * x[q].w);
            }
        }
        const float inv_l = (L > 0.f) ? 1.f / L : 0.f;
        uint4* dst = reinterpret_cast<uint4*>(
            a.o + (((size_t)b * a.Hq + hr) * a.Sq + row) * T::D_COLS + c16 * 16);
#pragma unroll
        for (int g8 = 0; g8 < 2; ++g8) {
            uint4 v;
            v.x = pack_bf16x2(acc[8 * g8 + 0] * inv_l, acc[8 * g8 + 1] * inv_l);
            v.y = pack_bf16x2(acc[8 * g8 + 2] * inv_l, acc[8 * g8 + 3] * inv_l);
            v.z = pack_bf16x2(acc[8 * g8 + 4] * inv_l, acc[8 * g8 + 5] * inv_l);
            v.w = pack_bf16x2(acc[8 * g8 + 6] * inv_l, acc[8 * g8 + 7] * inv_l);
            dst[g8] = v;
        }
        if (c16 == 0)
            a.lse[((size_t)b * a.Hq + hr) * a.Sq + row] =
                (L > 0.f) ? (M + lg2_approx(L)) * kLn2 : -INFINITY;
    }
}

// SPLIT: the instantiation can receive pieces of split units (only the
// unmasked, unwindowed one: the work split never cuts causal or windowed
// units, whose lengths differ); the others compile none of that code.
template <class T, bool SPLIT, bool VARLEN, bool EPI, bool PERSIST = false>
__device__ void prefill_correction_role(const CUtensorMap* tm_o, const PrefillArgs& a,
                                        const PrefillWork& w, PrefillAux<T>* aux, uint32_t tmem,
                                        uint32_t sQ, const WaitCtx& wc, unsigned long long* tr,
                                        int J0 = 0, int k = 0) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if ((warp & 3) != 0 || lane != 0) tr = nullptr;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const bool issuer = (warp & 3) == 0 && lane == 0;
    bool ok = true;
    for (int j = 0; j < w.n_max && ok; ++j) {
        for (int t = 0; t < T::NQ; ++t) {
            if (j >= w.n_kv[t]) continue;
            const int J = J0 + j;   // block index over the CTA's units
            if (!mbar_wait(smem_u32(&aux->bar_mb_full[sig_idx<T>(t, J)]), sig_par<T>(J), wc,
                           kErrWaitTimeout | kSiteCorrMbox)) {
                ok = false;
                break;
            }
            trace_mark(tr, kTrCorr, J0 + j, 4 * t);
            const float alpha = aux->mb_alpha[sig_idx<T>(t, J)][r];
            if (j > 0 && __any_sync(0xffffffffu, alpha < 1.f)) {
                // O_t must hold PV_t(j-1) before it is rebased
                if (!mbar_wait(smem_u32(&aux->bar_pv_done[sig_idx<T>(t, J - 1)]), sig_par<T>(J - 1), wc,
                               kErrWaitTimeout | kSiteCorrPv)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < T::D_COLS / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(lane_base + T::o_col(t) + c * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                    tmem_st32(lane_base + T::o_col(t) + c * 32, v);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive_warp(smem_u32(&aux->bar_p_ready[sig_idx<T>(t, J0 + j)]));   // O_t safe for PV_t(j)
            trace_mark(tr, kTrCorr, J0 + j, 4 * t + 1);
        }
    }
    // epilogue: O / row_sum -> bf16 -> shared (Q tile's space, 128-byte swizzled) -> TMA store
    for (int t = 0; t < T::NQ && ok; ++t) {
        const int nk = w.n_kv[t];
        if (!mbar_wait(smem_u32(&aux->bar_fin[t]), PERSIST ? (uint32_t)(k & 1) : 0u, wc,
                       kErrWaitTimeout | kSiteEpiMbox)) {
            ok = false;
            break;
        }
        trace_mark(tr, kTrCorr, J0 + w.n_max, 4 * t + 2);
        const float l = aux->mb_l[t][r];
        const float m = aux->mb_m[t][r];
        if (nk > 0) {
            // O is final once PV(nk-1) completed (value MMAs into one
            // accumulator complete in issue order).  The wait is exact: the
            // previous PV on the same barrier copy completed before the last
            // score MMA was issued.
            if (!mbar_wait(smem_u32(&aux->bar_pv_done[sig_idx<T>(t, J0 + nk - 1)]),
                           sig_par<T>(J0 + nk - 1), wc, kErrWaitTimeout | kSiteEpiPv)) {
                ok = false;
                break;
            }
            tc_fence_after();
        }
        if (SPLIT && w.piece >= 0) {
            // a piece of a split unit: unnormalised O, row max and row sum
            // -> this piece's scratch slot (merged below)
            float4* po = reinterpret_cast<float4*>(
                a.part_o + ((size_t)w.piece * T::NQ + t) * (T::D_COLS * T::BM));
#pragma unroll 1
            for (int c32 = 0; c32 < T::D_COLS / 32; ++c32) {
                uint32_t v[32];
                if (nk > 0) {
                    tmem_ld32(lane_base + T::o_col(t) + c32 * 32, v);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = 0u;
                }
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    po[(size_t)(c32 * 8 + q) * T::BM + r] =
                        make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                    __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
            }
            float* ml = a.part_ml + ((size_t)w.piece * T::NQ + t) * 2 * T::BM;
            ml[r] = (nk > 0) ? m : -INFINITY;
            ml[T::BM + r] = (nk > 0) ? l : 0.f;
            continue;
        }
        float lf, mf;
        const float inv_l = final_scale(a, w.h, l, m, lf, mf);
        if constexpr (PERSIST) {
            // persistent kernel: all of O, through the warp's staging
            // buffers and TMA stores (the Q tile's shared memory holds the
            // next unit's Q; the softmax warpgroup has gone on to that unit)
            const int row = w.row0 + t * T::BM + r;
            const int wrow = w.row0 + t * T::BM + (warp & 3) * 32;   // the warp's first row
            uint16_t* obase = a.o + (((size_t)w.b * a.Hq + w.h) * a.Sq + wrow) * (T::D_COLS * T::DV_SPLIT) + w.dv0;
            trace_wg(a, kTrCorr, J0 + w.n_max, 5);
            store_o_rows_staged<T, 2>(lane_base, T::o_col(t), obase, T::D_COLS * T::DV_SPLIT,
                                      a.Sq - wrow, nk, inv_l, EPI ? 2 * T::EPI_SPLIT : 0,
                                      (T::D_COLS + 31) / 32, stage_of<T>(sQ, warp), tm_o,
                                      w.dv0, wrow, w.b * a.Hq + w.h);
            trace_wg(a, kTrCorr, J0 + w.n_max, 6);
            if (nk > 0) {
                tc_fence_before();
                mbar_arrive_warp(smem_u32(&aux->bar_odrained));
            }
            if (row < a.Sq && (T::DV_SPLIT == 1 || w.dv0 == 0))
                a.lse[((size_t)w.b * a.Hq + w.h) * a.Sq + row] =
                    (lf > 0.f) ? (mf + lg2_approx(lf)) * kLn2 : -INFINITY;
            continue;
        }
        const uint32_t stage = sQ + t * T::QTILE;
        const int row = w.row0 + t * T::BM + r;
        // packed sequences: a tile that runs past the end of its sequence is
        // stored row by row (a TMA store would write the next sequence's rows)
        const bool direct = VARLEN && w.row0 + t * T::BM + T::BM > w.Lq;
        // chunks [0, EPI_SPLIT) are the softmax warpgroup's when split
        const int ch0 = (EPI && w.piece < 0) ? T::EPI_SPLIT : 0;
        if (VARLEN && direct) {
            constexpr int d_full = T::D_COLS * T::DV_SPLIT;
            uint16_t* orow = a.o + ((size_t)(w.q0 + row) * a.Hq + w.h) * d_full + w.dv0;
#pragma unroll 1
            for (int c32 = 0; c32 < (T::D_COLS + 31) / 32; ++c32) {
                uint32_t v[32];
                if (nk > 0) {
                    tmem_ld32(lane_base + T::o_col(t) + c32 * 32, v);
                    tmem_wait_ld();
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = 0u;
                }
#pragma unroll
                for (int g4 = 0; g4 < 4; ++g4) {
                    uint32_t pk[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        pk[e] = pack_bf16x2(__uint_as_float(v[g4 * 8 + 2 * e]) * inv_l,
                                            __uint_as_float(v[g4 * 8 + 2 * e + 1]) * inv_l);
                    if (row < w.Lq)
                        *reinterpret_cast<uint4*>(orow + c32 * 32 + g4 * 8) =
                            make_uint4(pk[0], pk[1], pk[2], pk[3]);
                }
            }
        } else {
            stage_o_rows<T>(lane_base, T::o_col(t), stage, r, nk, inv_l, 2 * ch0,
                            (T::D_COLS + 31) / 32);
        }
        // (with split output columns every part has the same statistics;
        // the first part stores LSE)
        if (row < (VARLEN ? w.Lq : a.Sq) && (T::DV_SPLIT == 1 || w.dv0 == 0)) {
            const float lse = (lf > 0.f) ? (mf + lg2_approx(lf)) * kLn2 : -INFINITY;
            if constexpr (VARLEN)
                a.lse[(size_t)w.h * a.total_q + w.q0 + row] = lse;   // [Hq, total_q]
            else
                a.lse[((size_t)w.b * a.Hq + w.h) * a.Sq + row] = lse;
        }
        fence_proxy_async_smem();
        mbar_arrive_warp(smem_u32(&aux->bar_epi[t]));
        if (issuer && !direct && w.row0 + t * T::BM < (VARLEN ? w.Lq : a.Sq) &&
            mbar_wait_lane(smem_u32(&aux->bar_epi[t]), 0, wc, kErrWaitTimeout | kSiteEpiStage)) {
#pragma unroll
            for (int ch = ch0; ch < T::OCH; ++ch)
                tma_store_3d(tm_o, stage + ch * T::CHUNK, w.dv0 + ch * 64,
                             (VARLEN ? w.q0 : 0) + w.row0 + t * T::BM,
                             VARLEN ? w.h : w.b * a.Hq + w.h);
            bulk_commit_group();
        }
        trace_mark(tr, kTrCorr, J0 + w.n_max, 4 * t + 3);
    }
    // the CTA may exit once the O stores have read shared memory
    if (issuer) bulk_wait_group_read_0();
    if (SPLIT && ok && w.piece >= 0) split_arrive<T>(a, w, aux, wc);
}

// --------------------------------------------------------------- kernel ----

template <int D, bool CAUSAL, bool WINDOW, bool VARLEN>
__global__ void __launch_bounds__(PrefillTraits<D>::THREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const PrefillArgs args) {
    using T = PrefillTraits<D>;
    static_assert(sizeof(PrefillAux<T>) <= T::SMEM_AUX, "auxiliary shared block too large");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sQ = (raw + 1023u) & ~1023u;   // 1024-aligned: swizzle atoms
    const uint32_t sRing = sQ + T::SMEM_Q;
    auto* aux = reinterpret_cast<PrefillAux<T>*>(smem_raw + (sQ - raw) + T::SMEM_Q + T::SMEM_RING);

    const int warp = threadIdx.x >> 5;
    const int wg = warp >> 2;
    const PrefillWork w = prefill_work<T, CAUSAL, WINDOW, VARLEN>(args, (int)blockIdx.x);

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&aux->bar_q), 1);
        for (int i = 0; i < T::NSLOT; ++i) {
            mbar_init(smem_u32(&aux->bar_full[i]), 1);
            mbar_init(smem_u32(&aux->bar_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&aux->bar_s_full[i]), 1);
        // warpgroup-to-warp signals: one elected arrive per warp
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&aux->bar_p_ready[i]), 8);   // 4 softmax + 4 correction warps
            mbar_init(smem_u32(&aux->bar_mb_full[i]), 4);
            mbar_init(smem_u32(&aux->bar_pv_done[i]), 1);
        }
        for (int t = 0; t < T::NQ; ++t) {
            mbar_init(smem_u32(&aux->bar_fin[t]), 4);
            mbar_init(smem_u32(&aux->bar_epi[t]), 4);
            mbar_init(smem_u32(&aux->bar_epi_sm[t]), 4);
        }
        mbar_init(smem_u32(&aux->bar_drain[0]), 1);
        mbar_init(smem_u32(&aux->bar_drain[1]), 1);
        mbar_init(smem_u32(&aux->bar_tail), 1);
        mbar_init(smem_u32(&aux->bar_split_a), 4);
        aux->abort_flag = 0;
        aux->merge_last = 0;
        mbar_fence_init();
    }
    if (warp == T::MMA_WARP) {
        tmem_alloc(smem_u32(&aux->tmem_base), T::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = aux->tmem_base;
    const WaitCtx wc{smem_u32(&aux->abort_flag), (uint32_t)args.wait_limit_ns, args.err_word};
    const int block_lin = blockIdx.x;
    unsigned long long* tr =
        (FA_PREFILL_TRACE && args.trace != nullptr && block_lin == args.trace_block) ? args.trace
                                                                                     : nullptr;

    if (wg < T::NQ) {
        setmaxnreg_inc<T::template Regs<CAUSAL || WINDOW>::SOFTMAX>();
        prefill_softmax_role<T, CAUSAL, WINDOW, VARLEN>(wg, &tm_o, args, w, aux, tmem, sQ, wc, tr);
    } else if (wg == T::CORR_WG) {
        setmaxnreg_dec<T::template Regs<CAUSAL || WINDOW>::CORR>();
        prefill_correction_role<T, !CAUSAL && !WINDOW && !VARLEN && T::DV_SPLIT == 1, VARLEN,
                                epi_split<T, CAUSAL || WINDOW, VARLEN>()>(&tm_o, args, w, aux,
                                                                          tmem, sQ, wc, tr);
    } else {
        setmaxnreg_dec<T::template Regs<CAUSAL || WINDOW>::OTHER>();
        if constexpr (T::CONSUME_ORDER) {
            if (warp == T::MMA_WARP)
                prefill_mma_role_dv<T>(args, w, aux, tmem, sQ, sRing, wc, tr);
            else if (warp == T::LOAD_WARP)
                prefill_load_role_dv<T, CAUSAL, WINDOW, VARLEN>(&tm_q, &tm_k, &tm_v, args, w, aux,
                                                                sQ, sRing, wc, tr);
        } else {
            if (warp == T::MMA_WARP)
                prefill_mma_role<T, VARLEN>(0, args, w, aux, tmem, sQ, sRing, wc, tr);
            else if (warp == T::LOAD_WARP)
                prefill_load_role<T, CAUSAL, WINDOW, VARLEN>(&tm_q, &tm_k, &tm_v, args, w, aux, sQ,
                                                             sRing, wc, tr);
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == T::MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, T::TMEM_COLS);
    }
    // the last piece of a split unit to arrive merges it, on all threads
    if (!CAUSAL && !WINDOW && !VARLEN && T::DV_SPLIT == 1 && aux->merge_last != 0 &&
        ld_volatile_shared(wc.abort_flag) == 0)
        merge_unit<T>(args, aux->merge_unit[0], aux->merge_unit[1], aux->merge_unit[2],
                      aux->merge_unit[3], (int)threadIdx.x, T::THREADS);
}

// ------------------------------------------------ persistent (head_dim 256) ----
//
// One CTA per SM walks a static list of units: unit i of CTA x is in wave i
// of the unit order, at position x in even waves and G - 1 - x in odd ones
// (G CTAs; a snake, so that with causal units, which come heaviest first,
// every CTA's total stays within one unit of the others').  Barriers, the
// ring, tensor memory and the score buffers stay live from one unit to the
// next: ring positions and key-block indices J count on over the CTA's units
// (only units with work count: kq numbers them), so every parity below is a
// running one.  What changes at a unit boundary:
//   * the producer loads the next unit's Q once the unit's last score MMA
//     has completed (bar_qfree), not once the unit is over;
//   * the correction warpgroup drains O to global memory through a 2 KB
//     staging area per warp and TMA stores (not through the Q tile's space,
//     which then already holds the next unit's Q) and arrives on
//     bar_odrained when done, while the softmax warpgroup goes on with the
//     next unit's scores;
//   * the first value MMA of the next unit, which overwrites O, waits for
//     bar_odrained; so does the softmax before it posts the next unit's
//     final statistics (their mailbox is read by the correction warpgroup
//     before it arrives);
//   * units without keys are written (O = 0, LSE of the sink or -inf) by the
//     correction warpgroup alone, without any signal.
__device__ __forceinline__ int persist_unit(int i, int x, int G) {
    return i * G + ((i & 1) ? G - 1 - x : x);
}

template <class T, bool CAUSAL, bool WINDOW>
__device__ void prefill_load_role_persist(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                          const CUtensorMap* tm_v, const PrefillArgs& a,
                                          PrefillAux<T>* aux, uint32_t sQ, uint32_t sRing,
                                          const WaitCtx& wc, unsigned long long* tr) {
    const int lane = threadIdx.x & 31;
    if (lane != 0) tr = nullptr;
    const int G = (int)gridDim.x, x = (int)blockIdx.x;
    const uint32_t bar_q = smem_u32(&aux->bar_q);
    if (lane == 0) {
        tma_prefetch_desc(tm_q);
        tma_prefetch_desc(tm_k);
        tma_prefetch_desc(tm_v);
    }
    int p = 0, ntail = 0, kq = 0;
    bool ok = true;
    for (int i = 0; ok; ++i) {
        const int u = persist_unit(i, x, G);
        if (u >= a.n_full) break;
        const PrefillWork w = prefill_work<T, CAUSAL, WINDOW, false>(a, u);
        if (w.n_max <= 0) continue;
        auto load = [&](int j, bool is_v, int pc) -> bool {
            return load_piece<T, false>(tm_k, tm_v, a, w, aux, sRing, wc, tr, j, is_v, pc, p,
                                        ntail);
        };
        // K_0 first: its slots are free while the previous unit's last
        // score MMA still reads Q
        for (int pc = 0; pc < T::PIECES && ok; ++pc) ok = load(0, false, pc);
        if (!ok) break;
        if (kq > 0 && !mbar_wait(smem_u32(&aux->bar_qfree), (uint32_t)((kq - 1) & 1), wc,
                                 kErrWaitTimeout | kSiteLoadQfree))
            break;
        if (lane == 0) {
            mbar_arrive_expect_tx(bar_q, (uint32_t)T::QTILE);
            load_chunks<T, T::NCH>(sQ, tm_q, 0, w.row0, w.b * a.Hq + w.h, bar_q);
            const int un = persist_unit(i + 1, x, G);   // this CTA's next unit
            if (un < a.n_full) prefetch_q_of<T, CAUSAL, WINDOW, false>(tm_q, a, un);
        }
        __syncwarp();
        ++kq;
        for (int j = 0; j < w.n_max && ok; ++j) {
            if (j + 1 < w.n_max)
                for (int pc = 0; pc < T::PIECES && ok; ++pc) ok = load(j + 1, false, pc);
            for (int pc = 0; pc < T::VPIECES && ok; ++pc) ok = load(j, true, pc);
        }
    }
    // every copy issued must have landed before the CTA exits
    if (lane == 0) {
        if (kq > 0) mbar_wait_drain(bar_q, (uint32_t)((kq - 1) & 1), a.wait_limit_ns);
        for (int q = p > T::NSLOT ? p - T::NSLOT : 0; q < p; ++q)
            mbar_wait_drain(smem_u32(&aux->bar_full[ring_slot<T>(q)]), ring_phase<T>(q),
                            a.wait_limit_ns);
    }
    __syncwarp();
}

// MMA issue over the CTA's units.  Block J of the CTA uses score buffer
// J & 1; S(J) waits for PV(J - 2), the last reader of that buffer's P, also
// across a unit boundary.
template <class T, bool CAUSAL, bool WINDOW>
__device__ void prefill_mma_role_persist(const PrefillArgs& a, PrefillAux<T>* aux, uint32_t tmem,
                                         uint32_t sQ, uint32_t sRing, const WaitCtx& wc,
                                         unsigned long long* tr) {
    const int lane = threadIdx.x & 31;
    if (lane != 0) {
        __syncwarp();
        return;
    }
    const int G = (int)gridDim.x, x = (int)blockIdx.x;
    const uint32_t qd0 = sdesc_lo_sw128(sQ, 16);
    const uint32_t kd0 = sdesc_lo_sw128(sRing, 16);
    const uint32_t vd0 = sdesc_lo_sw128(sRing, T::CHUNK);
    const uint32_t vd0r = sdesc_lo_sw128(sRing, T::VROW_CHUNK);   // row-split V slots
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t idesc_v = idesc_bf16_f32(128, T::PV_N, false, true);
    int p = 0;   // ring position of the next piece (the producer's order)
    auto next_piece = [&](unsigned site) -> bool {
        if (!mbar_wait_lane(smem_u32(&aux->bar_full[ring_slot<T>(p)]), ring_phase<T>(p), wc,
                            kErrWaitTimeout | site))
            return false;
        tc_fence_after();
        return true;
    };
    auto slot_desc = [&](uint32_t d0) { return d0 + (uint32_t)((ring_slot<T>(p) * T::SLOT) >> 4); };
    auto pv_done = [&](int J) -> bool {
        if (J < 0) return true;
        if (!mbar_wait_lane(smem_u32(&aux->bar_pv_done[sig_idx<T>(0, J)]), sig_par<T>(J), wc,
                            kErrWaitTimeout | kSiteMmaPv))
            return false;
        tc_fence_after();
        return true;
    };
    // S(J) = Q K^T into score buffer J & 1, each K piece released once its
    // K-steps complete
    auto score = [&](int J) -> bool {
        if (!pv_done(J - 2)) return false;
        trace_mark(tr, kTrMma, J, 0);
        for (int pc = 0; pc < T::PIECES; ++pc) {
            if (!next_piece(kSiteMmaK)) return false;
            trace_mark(tr, kTrMma, J, 1 + pc);
            const uint32_t kd = slot_desc(kd0);
#pragma unroll
            for (int kin = 0; kin < T::SLOT_CH * 4; ++kin) {
                const int kk = pc * T::SLOT_CH * 4 + kin;
                umma_ss_lo(tmem + T::s_col(J & 1), qd0 + kstep_off(kk), kd + kstep_off(kin),
                           idesc_s, kk > 0 ? 1u : 0u);
            }
            tc_commit(smem_u32(&aux->bar_empty[ring_slot<T>(p)]));
            ++p;
        }
        tc_commit(smem_u32(&aux->bar_s_full[J & 1]));
        return true;
    };
    int J0 = 0, kq = 0;
    bool ok = true;
    for (int i = 0; ok; ++i) {
        const int u = persist_unit(i, x, G);
        if (u >= a.n_full) break;
        const PrefillWork w = prefill_work<T, CAUSAL, WINDOW, false>(a, u);
        const int n = w.n_max;
        if (n <= 0) continue;
        if (!mbar_wait_lane(smem_u32(&aux->bar_q), (uint32_t)(kq & 1), wc,
                            kErrWaitTimeout | kSiteMmaQ))
            break;
        tc_fence_after();
        if (!score(J0)) break;
        if (n == 1) tc_commit(smem_u32(&aux->bar_qfree));
        for (int j = 0; j < n && ok; ++j) {
            const int J = J0 + j;
            if (j + 1 < n) {
                if (!score(J + 1)) {
                    ok = false;
                    break;
                }
                if (j + 2 == n) tc_commit(smem_u32(&aux->bar_qfree));   // Q no longer read
            }
            if (!mbar_wait_lane(smem_u32(&aux->bar_p_ready[sig_idx<T>(0, J)]), sig_par<T>(J), wc,
                                kErrWaitTimeout | kSiteMmaP)) {
                ok = false;
                break;
            }
            trace_mark(tr, kTrMma, J, 9);
            tc_fence_after();
            // the unit's first value MMA overwrites O: the previous unit's O
            // must have been read out
            if (j == 0 && kq > 0) {
                if (!mbar_wait_lane(smem_u32(&aux->bar_odrained), (uint32_t)((kq - 1) & 1), wc,
                                    kErrWaitTimeout | kSiteMmaOdrained)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            for (int nh = 0; nh < T::VPIECES; ++nh) {
                if (!next_piece(kSiteMmaV)) {
                    ok = false;
                    break;
                }
                trace_mark(tr, kTrMma, J, 10 + nh);
                issue_value_rows<T>(tmem + T::o_col(0), tmem + T::s_col(J & 1) + 64, nh,
                                    slot_desc(vd0r), idesc_v, j == 0);
                tc_commit(smem_u32(&aux->bar_empty[ring_slot<T>(p)]));
                ++p;
            }
            if (ok) tc_commit(smem_u32(&aux->bar_pv_done[sig_idx<T>(0, J)]));
        }
        J0 += n;
        ++kq;
    }
    {
        const uint32_t drain = smem_u32(&aux->bar_drain[0]);
        tc_commit(drain);
        mbar_wait_drain(drain, 0, a.wait_limit_ns);
    }
    __syncwarp();
}

// A unit without keys: O = 0 and LSE = log of the sink term (or -inf), by
// the correction warpgroup (thread = row).
template <class T>
__device__ void write_empty_unit(const PrefillArgs& a, const PrefillWork& w) {
    const int r = ((threadIdx.x >> 5) & 3) * 32 + (threadIdx.x & 31);
    const int row = w.row0 + r;
    float lf, mf;
    const float inv_l = final_scale(a, w.h, 0.f, -INFINITY, lf, mf);
    uint16_t* orow = a.o + (((size_t)w.b * a.Hq + w.h) * a.Sq + row) * T::D_COLS;
    store_o_rows_direct<T>(0u, 0u, orow, row < a.Sq, 0, inv_l, 0, T::D_COLS / 32);
    if (row < a.Sq)
        a.lse[((size_t)w.b * a.Hq + w.h) * a.Sq + row] =
            (lf > 0.f) ? (mf + lg2_approx(lf)) * kLn2 : -INFINITY;
}

template <int D, bool CAUSAL, bool WINDOW>
__global__ void __launch_bounds__(PrefillTraits<D>::THREADS, 1)
    prefill_kernel_persist(const __grid_constant__ CUtensorMap tm_q,
                           const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ CUtensorMap tm_o, const PrefillArgs args) {
    using T = PrefillTraits<D>;
    static_assert(T::NQ == 1 && T::DV_SPLIT == 1 && T::CONSUME_ORDER,
                  "persistent kernel: one Q tile, whole output columns, ring in consumption order");
    static_assert(sizeof(PrefillAux<T>) <= T::SMEM_AUX, "auxiliary shared block too large");
    // the correction warpgroup drains all of O: the softmax warpgroup goes
    // straight on to the next unit's first scores (measured: +0.8 % against
    // the drain split between the two warpgroups)
    constexpr bool EPI = false;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sQ = (raw + 1023u) & ~1023u;
    const uint32_t sRing = sQ + T::SMEM_Q;
    auto* aux = reinterpret_cast<PrefillAux<T>*>(smem_raw + (sQ - raw) + T::SMEM_Q + T::SMEM_RING);
    const int warp = threadIdx.x >> 5;
    const int wg = warp >> 2;

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&aux->bar_q), 1);
        for (int i = 0; i < T::NSLOT; ++i) {
            mbar_init(smem_u32(&aux->bar_full[i]), 1);
            mbar_init(smem_u32(&aux->bar_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&aux->bar_s_full[i]), 1);
            mbar_init(smem_u32(&aux->bar_p_ready[i]), 8);
            mbar_init(smem_u32(&aux->bar_mb_full[i]), 4);
            mbar_init(smem_u32(&aux->bar_pv_done[i]), 1);
        }
        mbar_init(smem_u32(&aux->bar_fin[0]), 4);
        mbar_init(smem_u32(&aux->bar_epi[0]), 4);
        mbar_init(smem_u32(&aux->bar_epi_sm[0]), 4);
        mbar_init(smem_u32(&aux->bar_drain[0]), 1);
        mbar_init(smem_u32(&aux->bar_drain[1]), 1);
        mbar_init(smem_u32(&aux->bar_tail), 1);
        mbar_init(smem_u32(&aux->bar_split_a), 4);
        mbar_init(smem_u32(&aux->bar_qfree), 1);
        mbar_init(smem_u32(&aux->bar_odrained), 4);   // the 4 correction warps
        aux->abort_flag = 0;
        aux->merge_last = 0;
        mbar_fence_init();
    }
    if (warp == T::MMA_WARP) {
        tmem_alloc(smem_u32(&aux->tmem_base), T::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = aux->tmem_base;
    const WaitCtx wc{smem_u32(&aux->abort_flag), (uint32_t)args.wait_limit_ns, args.err_word};
    unsigned long long* tr = (FA_PREFILL_TRACE && args.trace != nullptr &&
                              (int)blockIdx.x == args.trace_block)
                                 ? args.trace
                                 : nullptr;
    const int G = (int)gridDim.x, x = (int)blockIdx.x;

    if (wg == 0) {
        setmaxnreg_inc<T::template Regs<CAUSAL || WINDOW>::SOFTMAX>();
        int J0 = 0, kq = 0;
        for (int i = 0;; ++i) {
            const int u = persist_unit(i, x, G);
            if (u >= args.n_full || ld_volatile_shared(wc.abort_flag) != 0) break;
            const PrefillWork w = prefill_work<T, CAUSAL, WINDOW, false>(args, u);
            if (w.n_max <= 0) continue;
            prefill_softmax_role<T, CAUSAL, WINDOW, false, true>(0, &tm_o, args, w, aux, tmem, sQ,
                                                                 wc, tr, J0, kq);
            J0 += w.n_max;
            ++kq;
        }
    } else if (wg == T::CORR_WG) {
        setmaxnreg_dec<T::template Regs<CAUSAL || WINDOW>::CORR>();
        int J0 = 0, kq = 0;
        for (int i = 0;; ++i) {
            const int u = persist_unit(i, x, G);
            if (u >= args.n_full || ld_volatile_shared(wc.abort_flag) != 0) break;
            const PrefillWork w = prefill_work<T, CAUSAL, WINDOW, false>(args, u);
            if (w.n_max <= 0) {
                write_empty_unit<T>(args, w);
                continue;
            }
            prefill_correction_role<T, false, false, EPI, true>(&tm_o, args, w, aux, tmem, sQ, wc,
                                                                tr, J0, kq);
            J0 += w.n_max;
            ++kq;
        }
        // the epilogue's O stores must have read the staging area before exit
        if ((threadIdx.x & 31) == 0) bulk_wait_group_read_0();
    } else {
        setmaxnreg_dec<T::template Regs<CAUSAL || WINDOW>::OTHER>();
        if (warp == T::MMA_WARP)
            prefill_mma_role_persist<T, CAUSAL, WINDOW>(args, aux, tmem, sQ, sRing, wc, tr);
        else if (warp == T::LOAD_WARP)
            prefill_load_role_persist<T, CAUSAL, WINDOW>(&tm_q, &tm_k, &tm_v, args, aux, sQ, sRing,
                                                         wc, tr);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == T::MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, T::TMEM_COLS);
    }
}

}  // namespace fa

#include "prefill_wide.cuh"

namespace fa {

// Host-side launch of one head-dimension instantiation.
using PrefillKernelFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, PrefillArgs);

template <int D, bool VARLEN>
PrefillKernelFn pick_prefill_kernel(bool causal, bool window) {
    return window ? (causal ? prefill_kernel<D, true, true, VARLEN> : prefill_kernel<D, false, true, VARLEN>)
                  : (causal ? prefill_kernel<D, true, false, VARLEN>
                            : prefill_kernel<D, false, false, VARLEN>);
}

template <int D>
cudaError_t launch_prefill_impl(const PrefillLaunch& p, cudaStream_t stream) {
    using T = PrefillTraits<D>;
    const bool window = p.args.window > 0;
    if constexpr (D == 256) {
        // dense launches of whole units: one persistent CTA per SM
        if (p.args.cu_seqlens_q == nullptr && p.n_tail == 0 && p.num_sms > 0 && p.args.n_full > 0) {
            const PrefillKernelFn kern =
                window ? (p.causal ? prefill_kernel_persist<D, true, true>
                                   : prefill_kernel_persist<D, false, true>)
                       : (p.causal ? prefill_kernel_persist<D, true, false>
                                   : prefill_kernel_persist<D, false, false>);
            cudaError_t e = cudaFuncSetAttribute(
                kern, cudaFuncAttributeMaxDynamicSharedMemorySize, T::SMEM_TOTAL);
            if (e != cudaSuccess) return e;
            const unsigned grid = (unsigned)min(p.args.n_full, p.num_sms);
            // (the persistent kernel stores O through its 32 x 32 map)
            kern<<<grid, T::THREADS, T::SMEM_TOTAL, stream>>>(p.tm_q, p.tm_k, p.tm_v, p.tm_o32,
                                                              p.args);
            return cudaGetLastError();
        }
    }
    if constexpr (D == 96 || D == 128) {
        // dense, no window: 256-key score blocks, one persistent CTA per SM
        if (p.wide) {
            using W = WideTraits<D>;
            // (head-packed GQA tiles, and units split along the keys: instances
            // of their own; split launches are never causal)
            const bool split = p.n_tail > 0;
            const PrefillKernelFn kern =
                split ? (p.args.pack > 1 ? prefill_kernel_wide<D, false, true, true>
                                         : prefill_kernel_wide<D, false, false, true>)
                : p.args.pack > 1
                    ? (p.causal ? prefill_kernel_wide<D, true, true, false>
                                : prefill_kernel_wide<D, false, true, false>)
                    : (p.causal ? prefill_kernel_wide<D, true, false, false>
                                : prefill_kernel_wide<D, false, false, false>);
            cudaError_t e = cudaFuncSetAttribute(
                kern, cudaFuncAttributeMaxDynamicSharedMemorySize, W::SMEM_TOTAL);
            if (e != cudaSuccess) return e;
            const unsigned grid = (unsigned)min(p.args.n_work, p.num_sms);
            kern<<<grid, W::THREADS, W::SMEM_TOTAL, stream>>>(p.tm_q, p.tm_k, p.tm_v, p.tm_o32,
                                                              p.args);
            return cudaGetLastError();
        }
    }
    const PrefillKernelFn kern = p.args.cu_seqlens_q != nullptr
                                     ? pick_prefill_kernel<D, true>(p.causal, window)
                                     : pick_prefill_kernel<D, false>(p.causal, window);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         T::SMEM_TOTAL);
    if (e != cudaSuccess) return e;
    const unsigned grid =
        ((unsigned)p.args.n_full + (unsigned)p.n_tail * (unsigned)p.args.split) * T::DV_SPLIT;
    kern<<<grid, T::THREADS, T::SMEM_TOTAL, stream>>>(p.tm_q, p.tm_k, p.tm_v, p.tm_o, p.args);
    return cudaGetLastError();
}

}  // namespace fa
