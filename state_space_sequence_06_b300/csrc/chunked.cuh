// Chunked prefill on the tensor cores: tcgen05 MMAs with TMEM accumulators,
// inputs staged by TMA.
//
// The recurrence ("Together AI announces Mamba-3", sections 1-3: an
// exponential-trapezoid update of a complex state applied as a rotation,
// SISO or rank-R MIMO) is evaluated chunk by chunk.  The Mamba-2
// state-space/attention duality (same page, history table) turns each
// chunk into dense products.  Inside a chunk of Q tokens, with chunk-local
// cumulative log-decay Lam_i = sum_{s<=i} dt_s A and angle phi_i[k] =
// sum_{s<=i} dt_s theta_s[k], and psi_i = phi_end - phi_i:
//
//   Bt_j = Bhat_j e^{-i Phi_j},  Ct_t = Chat_t e^{-i Phi_t}   (rotations, f16)
//   S    = Re(Ct Bt^H)    = realified Ct . Bt^T                (MMA 1)
//   S'   = S * e^{Lam_t - Lam_j} * w_tj  for j <= t, else 0
//          w_tt = lam_t dt_t,  w_tj = lam_j dt_j + (1 - lam_{j+1}) dt_{j+1}
//   Y    = S' X                                                (MMA 2)
//        + e^{Lam_t} Re(Ct^H G')                               (MMA 3)
//        + D x
//   G'   <- e^{Lam_end} G' + Bt^T (W X),  W_j = e^{Lam_end - Lam_j} w'_j   (MMA 4)
//
// Phi_j is the cumulative angle from the start of the sequence, kept
// reduced modulo 2 pi per pair (the chunk-local sum is added to a running
// phase once per chunk), so the state G' lives in the rotating frame
// e^{-i Phi}: the rotation of the state between chunks costs nothing and
// only the final state is turned back.  w'_j = lam_j dt_j + (1 - lam_{j+1})
// dt_{j+1} includes the next token's trapezoid coefficient (zero past the
// end of the sequence), so the state carried between chunks already holds
// the next token's previous-token term.  Decays are chunk-local and taken
// as exponentials of differences (or as a product of two factors when the
// chunk's log-decay range keeps both inside f32), so nothing overflows at
// any sequence length.
//
// One CTA walks the chunks of one (sequence, head) unit and keeps the f32
// state in TMEM for the whole sequence: the state never travels through
// HBM between chunks.  Operands are f16 with f32 accumulation; bf16 inputs
// convert exactly.  The rotated B and C, the masked and weighted scores S'
// and the weighted inputs W X are each carried as a pair hi + lo of f16
// values (hi = f16(v), lo = f16(v - hi)), and every product takes the
// hi*hi, hi*lo and lo*hi terms, so those operands keep about 21 bits: one
// f16 rounding (11 bits) is not enough for outputs 20-40x the rms of y,
// which the tails of the dt distribution produce.  Only the state copy R
// that feeds the inter-chunk output stays a single f16.  S' is written
// over its own scores in TMEM (each 16-column block of f32 S becomes 8
// columns of packed f16 hi words and 8 of lo words) and read from there by
// MMA 2 as its A operand; inside each block of 16 K rows, MMA 2 sees the
// columns of S' in the order kperm gives, and the f16 copy of X takes its
// rows in the same order.
#pragma once

#include <cuda.h>  // CUtensorMap and its enums (types only: the driver entry point is looked up at run time)

#include "common.cuh"
#include "umma.cuh"

namespace m3 {

struct ChunkParams {
  const __nv_bfloat16* x;
  const __nv_bfloat16* B;
  const __nv_bfloat16* dt;
  const __nv_bfloat16* lam;
  const float* A;
  const float* D;
  const int32_t* cu_seqlens;  // NULL: fixed length L per batch row
  // one CTA per unit with packed sequences: CTA b runs head b % H of
  // sequence seq_order[b / H] (longest sequences first), or unit b when NULL
  const int32_t* seq_order;
  void* y;                  // f32, or bf16 when ybf
  int ybf;
  float* h;                 // state slots or NULL
  __nv_bfloat16* prev_B;    // carry slots or NULL
  __nv_bfloat16* prev_x;
  int64_t L;
  int H;
  int G;  // B and C groups (head h uses group h / (H / G))
  int pro;               // m3_prologue flags
  const float* dt_bias;  // [H] or NULL
  // Balanced schedule (bal_grid == 0: one CTA per (sequence, head) unit).
  // With fixed-length sequences the bal_units units' chunks, unit after
  // unit, are cut into bal_grid equal ranges, one per CTA (all resident at
  // once: a cooperative launch).  A unit cut by the boundary before CTA k is
  // a prefill of its first chunks in CTA k - 1 (run first there) followed by
  // a prefill of the rest in CTA k (run last there) from the state and carry
  // handed over through slot k.
  int bal_grid;
  int bal_units;
  float* xh;             // handover h [slot][K2][P][2]
  __nv_bfloat16* xB;     // handover carry [slot][R][N]
  __nv_bfloat16* xx;     // handover carry [slot][R][P]
  int* xflag;            // [slot]: 1 once the slot is written (zeroed before the launch)
  // Test hooks (both 0 in normal use): the bounded-wait limit in ns (0:
  // kWaitLimitNs), and a planted fault (m3_test_fault):
  // M3_TEST_FAULT_SKIP_HANDOVER_RELEASE makes the writers of the handover
  // slots leave their flags unset, so the readers' waits run out.
  unsigned long long wait_ns;
  int fault;
  // Split schedule (split_grid > 0): the units' chunks, unit after unit,
  // are cut into split_grid equal ranges, CTA k running range k: the end of
  // one unit and the start of the next at most (split_pieces), piece i in
  // handover slot 2k + i.  The state-only pass (the kernel's SO variant)
  // runs every piece that does not end its unit from the zero state with the
  // carry of its previous token, and writes the piece's own final state to
  // seg_h and its total decay and rotation e^{Lam + i Phi} per pair to
  // seg_alpha; the full pass then runs every piece from its exact initial
  // state (its slot, combined from those on the device), and only the piece
  // that ends a unit writes the caller's state.
  int split_grid;
  float* seg_h;         // [slot][K2][P][2]
  float2* seg_alpha;    // [slot][K2]
};


constexpr int kMaxSeg = 8;  // segments per CTA in a balanced schedule
// SEG_SPLIT: a piece of the split schedule: its carry is the previous
// token's own B and x rows (at a unit's start the caller's carry, which
// the full pass reads from a copy in the piece's slot: the unit's last
// piece overwrites the caller's), and its slot is ready when the kernel
// starts (no flag to wait for)
constexpr int SEG_SRC_SLOT = 1, SEG_DST_SLOT = 2, SEG_NO_FINAL = 4, SEG_SPLIT = 8;

// Split schedule: range k of `grid` equal ranges of the units' `total`
// chunks (nch per unit, unit after unit), as at most two pieces {unit, first
// chunk, end chunk} within their units (a range is never longer than a unit:
// the schedule runs with grid >= units).  Returns the number of pieces.
__host__ __device__ inline int split_pieces(int64_t nch, int64_t total, int grid, int k, int3 piece[2]) {
  const int64_t lo = (int64_t)k * total / grid, hi = (int64_t)(k + 1) * total / grid;
  int n = 0;
  for (int64_t u = lo / nch; u * nch < hi && n < 2; ++u) {
    const int64_t cb = lo > u * nch ? lo : u * nch, ce = hi < (u + 1) * nch ? hi : (u + 1) * nch;
    if (cb < ce) piece[n++] = make_int3((int)u, (int)(cb - u * nch), (int)(ce - u * nch));
  }
  return n;
}

__host__ __device__ constexpr int align_up(int v, int a) { return (v + a - 1) / a * a; }

// RE: theta = 0 (a real state, the Mamba-2 special case): B and C need no
// rotation, convert to f16 exactly and carry no lo parts, and theta is not
// loaded.
template <int N_, int R_, int Q_, bool RE_ = false>
struct ChunkCfg {
  static constexpr bool RE = RE_;
  static constexpr int N = N_, R = R_, Q = Q_, P = 64;
  static constexpr int K2 = N / 2;  // complex pairs
  static constexpr int MR = Q * R;  // rows of S and Y: (token, rank)
  static_assert(MR == 64, "Q*R must be 64 (S and the outputs are double-buffered in TMEM)");
  static_assert(N == 64 || N == 128, "N must be 64 or 128");
  // warp roles: prologue warps (16 for SISO, 8 for MIMO, whose per-thread
  // state is larger), 4 state/output warps, then one warp each for the
  // intra-chunk MMAs (1 and 2), the TMA loads and the state-chain MMAs (4
  // and 3).  The prologue's work is latency-bound: more warps hide more of it.
  static constexpr int NPRO = R == 1 ? 512 : 256, NSTA = 128, NT = NPRO + NSTA + 96;
  static constexpr int W_STA = NPRO / 32, W_MMA = W_STA + NSTA / 32, W_TMA = W_MMA + 1, W_MMA2 = W_TMA + 1;

  // rotation work split: consecutive threads take consecutive pairs (so
  // shared-memory rows are read without bank conflicts), G token groups
  static constexpr int G = NPRO / K2, TPG = Q / G;
  static_assert(NPRO % K2 == 0 && Q % G == 0, "angle-scan split");
  // one chunk stage.  TMA writes bf16 C and B straight into their (hi)
  // 128B-swizzled operand tiles, which the prologue rotates and converts to
  // f16 in place; x lands in the tile that then receives (W X) hi, theta in
  // the area that then receives (W X) lo when it is large enough.
  static constexpr int CT_BYTES = MR * N * 2;  // C, B tiles: [N/64 blocks][MR rows][128 B]
  static constexpr int XT_BYTES = MR * P * 2;  // X, WX tiles: [MR rows][128 B]
  static constexpr int TH_BYTES = Q * K2 * 2;  // theta [Q][K2] bf16 (unswizzled)
  // B hi and lo are interleaved per 64-column block (block kb: hi at
  // OFF_B + kb * BB, lo MR rows after it)
  static constexpr int OFF_C = 0, OFF_CLO = CT_BYTES, OFF_B = 2 * CT_BYTES, OFF_BLO = OFF_B + MR * 128;
  static constexpr int BB = 2 * MR * 128;  // bytes between B blocks
  static constexpr int OFF_X = 4 * CT_BYTES;  // x (bf16), then (W X) hi
  static constexpr int OFF_TH = OFF_X + XT_BYTES;
  static constexpr bool WXLO_IN_TH = TH_BYTES >= XT_BYTES;
  static constexpr int OFF_WXLO = WXLO_IN_TH ? OFF_TH : align_up(OFF_TH + TH_BYTES, 1024);
  static constexpr int STAGE = align_up(WXLO_IN_TH ? OFF_TH + TH_BYTES : OFF_WXLO + XT_BYTES, 1024);
  static constexpr uint32_t STAGE_TX = 2 * CT_BYTES + XT_BYTES + (RE ? 0 : TH_BYTES);
  // outside the stages: X in f16 (it lives until the output of its chunk,
  // so it and the per-chunk scalars rotate through XB slots: three when they
  // fit) and R (MN-major); S' lives in TMEM
  static constexpr int RT_BYTES = N * P * 2;
  static constexpr int smem_for(int ns, int xb) { return ns * STAGE + xb * XT_BYTES + RT_BYTES + 1024; }
  static constexpr int STATIC_EST = 3 * 6 * Q * 4 + (NPRO / K2) * K2 * 4 + 2048;  // scalars, scan, misc
  static constexpr int XB = smem_for(2, 3) + STATIC_EST <= 232448 ? 3 : 2;
  // stages of the full pass: three at rank 1 when they fit (N = 64), else
  // two (at rank 4 a third stage measured slower: the prologue runs further
  // ahead of the state warps, the tighter role there)
  static constexpr int NSF = R == 1 && smem_for(3, XB) + STATIC_EST <= 232448 ? 3 : 2;
  static constexpr int OFF_XB = NSF * STAGE;
  static constexpr int OFF_RT = OFF_XB + XB * XT_BYTES;
  static constexpr int SMEM = OFF_RT + RT_BYTES + 1024;  // + alignment slack
  // state-only pass: a stage without its C tiles (from the B tiles on)
  static constexpr int SO_STRIDE = STAGE - OFF_B;
  static_assert(SMEM + STATIC_EST <= 232448, "shared memory of one CTA");
  // TMEM columns (f32): S[2] (then S' in place), Y[2], Yi[2], state, chunk-local state
  static constexpr int COL_S = 0, COL_Y = 2 * MR, COL_YI = 2 * MR + 2 * P, COL_G = 2 * MR + 4 * P;
  static constexpr int COL_SC = COL_G + P;  // the chunk-local state B^T (W X) of MMA 4
  // its second buffer in the state-only pass, which has no S, Y or Yi
  static constexpr int COL_SC1 = COL_S;
  static constexpr int TMEM_COLS = 512;
  static_assert(COL_SC + P <= TMEM_COLS, "TMEM columns");
};

// TMEM lane holding row `row` of an M-row accumulator (M = 64 uses lanes
// 0-15 of each 32-lane quarter; M = 128 uses lane = row).
__device__ __forceinline__ int acc_row_of(int M, int quarter, int lane) {
  return M == 128 ? 32 * quarter + lane : (lane < 16 ? 16 * quarter + lane : -1);
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// v = hi + lo with hi = f16(v) and lo = f16(v - hi), both returned packed as half2.
__device__ __forceinline__ void split_half2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 hf = __half22float2(h);
  const __half2 l = __floats2half2_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

__device__ __forceinline__ float2 bf2_to_f2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

// Row of the f16 copy of X that holds row j of X.  Inside each block of 16
// rows it is the K position at which MMA 2 reads column j of S' from TMEM:
// S -> S' stores the columns 8 g + 2 m + e (g, e < 2, m < 4) of a block as
// the f16 pair of word column 2 m + g, which holds K positions 4 m + 2 g + e.
__host__ __device__ constexpr int kperm(int j) {
  return (j & ~15) | (((j & 7) >> 1) << 2) | (((j >> 3) & 1) << 1) | (j & 1);
}

// sin and cos of x after one reduction step by 2*pi (|x| stays within a few
// tens of radians here), on the special-function unit.
__device__ __forceinline__ void sincos_reduced(float x, float* s, float* c) {
  const float n = rintf(x * 0.15915494309189535f);
  __sincosf(fmaf(-n, 6.283185307179586f, x), s, c);
}

constexpr uint32_t kMaxPolls = 1u << 22;
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;  // 200 ms: far beyond any legitimate wait

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Per-CTA abort record in shared memory: the flag that the first role to
// give up a wait sets, and this launch's wait limit.
struct CtaAbort {
  int flag;
  int pad;
  unsigned long long limit_ns;
};

// Bounded wait.  Gives up (and makes every role of this CTA give up) when
// the phase has not completed within the launch's limit (200 ms unless a
// test asks for less), or as soon as another role of this CTA has recorded
// a failure, so a stalled pipeline ends each CTA within a fraction of a
// second with M3_ERR_TIMEOUT.  Waiting threads read nothing outside their
// own CTA: a poll of a global word by every waiting warp of every CTA costs
// memory requests the pipeline needs.
//
// Only the first poll is inlined at each call site; the loop is one shared
// out-of-line copy.  The kernel's roles run different code at the same time
// on one SM, and instruction fetch is a shared resource: every copy of code
// that is executed each chunk costs instruction-cache capacity.
__device__ __noinline__ bool wait_or_abort_slow(uint32_t bar, uint32_t parity, volatile CtaAbort* ab) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1; i < kMaxPolls; ++i) {
    if (umma::mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0) {
      if (ab->flag) return false;
      if (globaltimer_ns() - t0 > ab->limit_ns) break;
    }
  }
  ab->flag = 1;
  atomicExch(&g_status, (int)M3_ERR_TIMEOUT);
  return false;
}
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile CtaAbort* ab) {
  if (umma::mbar_try_wait(bar, parity)) return true;
  return wait_or_abort_slow(bar, parity, ab);
}

// SO: the state-only pass of the split schedule: no C, no scores, no
// outputs; MMA 4 and the state chain only, each segment's final state and
// total decay and rotation to seg_h / seg_alpha.
// XC: the prologue warps convert X to f16 and form W X (the full pass at
// rank 1), instead of the state warps.
template <int N, int R, int Q, bool RE, bool SO = false, bool XC = false>
__global__ void __launch_bounds__(ChunkCfg<N, R, Q, RE>::NT, 1)
    chunked_prefill_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_B,
                           const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_th,
                           const ChunkParams p) {
  using Cfg = ChunkCfg<N, R, Q, RE>;
  constexpr int P = Cfg::P, K2 = Cfg::K2, MR = Cfg::MR, NPRO = Cfg::NPRO, NSTA = Cfg::NSTA;
  constexpr int G = Cfg::G, TPG = Cfg::TPG, XB = Cfg::XB;
  using namespace umma;

  extern __shared__ uint8_t smem_raw[];
  // barriers: full (TMA landed), phend (the phase after the chunk written,
  // read where a segment ends), opready (prologue done), free (stage no longer
  // read by MMAs), xready (X of the slot's chunk converted), xfree (X slot and
  // output accumulators no longer read), sfull (MMA 1 done), yfull (MMAs 2
  // and 3 done), spready (S' of the buffer written), scfull (MMA 4 done: the chunk-local
  // state is in TMEM), scfree (the state warps have folded it into the
  // state), stready (R, the f16 copy of the state for MMA 3, written; once
  // before the first chunk and once per chunk), rfree (MMA 3 done reading
  // R).  A phase-parity wait is only sound when the waiter can never fall two
  // phases behind the barrier; each pairing below is chained so that it
  // cannot.
  // (full, opready and free per stage: NS of them)
  __shared__ __align__(8) uint64_t bar_full[3], bar_opready[3], bar_free[3], bar_sfull[2], bar_yfull[2], bar_spready[2];
  __shared__ __align__(8) uint64_t bar_xfree[XB], bar_xready[XB], bar_phend[XB];
  __shared__ __align__(8) uint64_t bar_stready, bar_rfree;
  // scfull / scfree per chunk-local state buffer: one buffer (index 0) in the
  // full pass; two in the state-only pass, chunk c in buffer c & 1, so MMA 4
  // of chunk c + 1 does not wait for the state step of chunk c
  __shared__ __align__(8) uint64_t bar_scfull[2], bar_scfree[2];
  // mdone[i]: every product MMA thread i issued is complete (its last commit,
  // waited for before the TMEM is freed, also after an abort)
  __shared__ __align__(8) uint64_t bar_mdone[2];
  __shared__ uint32_t tmem_base_s;
  __shared__ CtaAbort s_abort;  // this CTA's abort flag and wait limit
  // per-chunk scalars, one set per X slot (chunk c uses slot c % XB)
  __shared__ float sLam[XB][Q], sELam[XB][Q], sGam[XB][Q], sWp[XB][Q], sDw[XB][Q], sLamEnd[XB];
  __shared__ __align__(16) float sBw[XB][Q];
  // prologue scratch
  __shared__ float sDt[Q + 1], sBet[Q + 1], sWarpTot[4];
  __shared__ float sPsum[G][K2];
  // cumulative angle per pair at the start of chunk c, in [-pi, pi): buffer c & 1
  // (chunk c writes the next chunk's while others may still read its own)
  __shared__ float sPhi[2][K2];
  __shared__ float sBScl[MR], sCScl[MR];  // BC norm: 1 / rms of each (token, rank) row of the tile
  __shared__ float sCarryScl[8];          // BC norm of the carried B rows at a segment start
  __shared__ __nv_bfloat16 sCarryX[R * 64];  // the carried x rows at a segment start
  __shared__ float sPhiEndX[XB][K2];  // the same after chunk c (slot c % XB), for the state warps

  // this CTA's segments: {unit, first token, end token, flags}, the first
  // chunk of each in the CTA's chunk stream, and the first token's row
  __shared__ int4 sSeg[kMaxSeg];
  __shared__ int sSegC0[kMaxSeg + 1];
  __shared__ long long sSegTok0[kMaxSeg];
  __shared__ int sSegHead[kMaxSeg];
  __shared__ float sSegA[kMaxSeg], sSegD[kMaxSeg];  // the head's A and D (read once, not per chunk)
  __shared__ int sNseg;

  uint8_t* sm = smem_raw + ((1024u - (saddr(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int H = p.H;
  if (tid == 0) {
    int ns = 0;
    if (p.bal_grid) {
      const int64_t nch = (p.L + Q - 1) / Q, total = (int64_t)p.bal_units * nch;
      const int k = blockIdx.x;
      const int64_t lo = k * total / p.bal_grid, hi = (k + 1) * total / p.bal_grid;
      // head: the first part of a unit whose rest CTA k + 1 runs (first here);
      // tail: the rest of a unit CTA k - 1 started (last here)
      int4 head_seg = make_int4(0, 0, 0, -1), tail_seg = make_int4(0, 0, 0, -1);
      int4 mid[kMaxSeg];
      int nmid = 0;
      for (int64_t u = lo / nch; u * nch < hi; ++u) {
        const int64_t cb = lo > u * nch ? lo : u * nch, ce = hi < (u + 1) * nch ? hi : (u + 1) * nch;
        const int tb = (int)((cb - u * nch) * Q);
        const int te = (int)((ce - u * nch) * Q < p.L ? (ce - u * nch) * Q : p.L);
        int4 sg = make_int4((int)u, tb, te, 0);
        if (cb > u * nch) {
          sg.w = SEG_SRC_SLOT | (k << 8);
          tail_seg = sg;
        } else if (ce < (u + 1) * nch) {
          sg.w = SEG_DST_SLOT | ((k + 1) << 8);
          head_seg = sg;
        } else if (nmid < kMaxSeg - 2) {  // (the host keeps a CTA's whole units to kMaxSeg - 2)
          mid[nmid++] = sg;
        }
      }
      if (head_seg.w >= 0) sSeg[ns++] = head_seg;
      for (int i = 0; i < nmid; ++i) sSeg[ns++] = mid[i];
      if (tail_seg.w >= 0) sSeg[ns++] = tail_seg;
    } else if (p.split_grid) {
      // this CTA's pieces; every one starts from the zero state in the
      // state-only pass and from its handover slot (the combined state) in
      // the full pass, with the carry of the token before it in both
      const int64_t nch = (p.L + Q - 1) / Q;
      int3 pc[2];
      const int np = split_pieces(nch, (int64_t)p.bal_units * nch, p.split_grid, blockIdx.x, pc);
      for (int i = 0; i < np; ++i) {
        const bool ends_unit = pc[i].z == nch;
        if (SO && ends_unit) continue;  // its own final state is needed by no later piece
        const int tb = pc[i].y * Q, te = (int)((int64_t)pc[i].z * Q < p.L ? (int64_t)pc[i].z * Q : p.L);
        int fl = ((2 * (int)blockIdx.x + i) << 8) | SEG_SRC_SLOT | SEG_SPLIT;
        if (SO)
          fl |= SEG_DST_SLOT;
        else if (!ends_unit)
          fl |= SEG_NO_FINAL;
        sSeg[ns++] = make_int4(pc[i].x, tb, te, fl);
      }
    } else {
      const int u = p.seq_order ? p.seq_order[blockIdx.x / H] * H + (int)blockIdx.x % H : (int)blockIdx.x;
      const int sq = u / H;
      const int n = p.cu_seqlens ? p.cu_seqlens[sq + 1] - p.cu_seqlens[sq] : (int)p.L;
      if (n > 0) sSeg[ns++] = make_int4(u, 0, n, 0);
    }
    int c0 = 0;
    for (int i = 0; i < ns; ++i) {
      const int sq = sSeg[i].x / H;
      const long long base = p.cu_seqlens ? (long long)p.cu_seqlens[sq] : (long long)sq * p.L;
      sSegTok0[i] = base + sSeg[i].y;
      sSegHead[i] = sSeg[i].x % H;
      sSegA[i] = p.A[sSeg[i].x % H];
      sSegD[i] = p.D[sSeg[i].x % H];
      sSegC0[i] = c0;
      c0 += (sSeg[i].z - sSeg[i].y + Q - 1) / Q;
    }
    sSegC0[ns] = c0;
    sNseg = ns;
  }
  __syncthreads();
  const int nseg = sNseg;
  const int nchunks = sSegC0[nseg];
  if (nchunks == 0) return;  // nothing to do; the state slot keeps its contents
  // segment of chunk c of this CTA's stream (a handful of entries)
  // (from segment si0 on: the roles walk their chunks in order, so the
  // segment they were last in is where the search starts)
  auto seg_from = [&](int c, int si0) {
    int si = si0;
    while (si + 1 < nseg && c >= sSegC0[si + 1]) ++si;
    return si;
  };
  auto seg_of = [&](int c) { return seg_from(c, 0); };
  auto seg_head = [&](int si) { return sSegHead[si]; };
  auto seg_ntok = [&](int si) { return (int64_t)(sSeg[si].z - sSeg[si].y); };
  auto seg_last = [&](int c) { return c + 1 == sSegC0[seg_of(c) + 1]; };
  volatile CtaAbort* abort_flag = &s_abort;
  constexpr bool xc_pro = XC && !SO && R == 1;

  uint8_t* Rt = sm + Cfg::OFF_RT;
  // Stages: in the full pass three at rank 1 with N = 64, else two; three
  // in the state-only pass, whose stages hold no C tiles (stage s there
  // starts OFF_B bytes before its B tiles, which follow the previous
  // stage's last tile; its C offsets are unused).
  constexpr int NS = SO ? 3 : Cfg::NSF;
  static_assert(!SO || 3 * Cfg::SO_STRIDE <= Cfg::SMEM - 1024, "three state-only stages");
  auto stage = [&](int s) { return SO ? sm + s * Cfg::SO_STRIDE - Cfg::OFF_B : sm + s * Cfg::STAGE; };
  auto xbuf = [&](int x) { return sm + Cfg::OFF_XB + x * Cfg::XT_BYTES; };
  // has the output of chunk cc (and its MMA 2) released X slot cc % XB?
  auto wait_xfree = [&](int cc) {
    return wait_or_abort(saddr(&bar_xfree[cc % XB]), (uint32_t)((cc / XB) & 1), abort_flag);
  };

  if (tid == 0) {
    s_abort.flag = 0;
    s_abort.limit_ns = p.wait_ns ? p.wait_ns : kWaitLimitNs;
    for (int s = 0; s < 3; ++s) {
      mbar_init(saddr(&bar_full[s]), 1);
      mbar_init(saddr(&bar_opready[s]), 1);
      mbar_init(saddr(&bar_free[s]), SO ? 1 : 2);   // MMA 1 and MMAs 4/3 completions (SO: MMA 4)
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(saddr(&bar_sfull[s]), 1);
      mbar_init(saddr(&bar_yfull[s]), 2);  // MMA 2 and MMA 3 completions
      mbar_init(saddr(&bar_spready[s]), NPRO);  // every prologue thread (one arrival per warp of 32)
    }
    for (int x = 0; x < XB; ++x) {
      // MMA 2 completion and the output epilogue (SO: the state warps, once
      // the slot's scalars are no longer read)
      mbar_init(saddr(&bar_xfree[x]), SO ? 1 : 2);
      mbar_init(saddr(&bar_xready[x]), 1);  // X converted (state or prologue warps; not in SO)
      mbar_init(saddr(&bar_phend[x]), K2);  // the phase after the slot's chunk, one arrival per pair
    }
    mbar_init(saddr(&bar_stready), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(saddr(&bar_scfull[b]), 1);
      mbar_init(saddr(&bar_scfree[b]), 1);
    }
    mbar_init(saddr(&bar_rfree), 1);
    mbar_init(saddr(&bar_mdone[0]), 1);
    mbar_init(saddr(&bar_mdone[1]), 1);
    mbar_init_fence();
  }
  if (warp == 0) {
    tmem_alloc(saddr(&tmem_base_s), Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  if (warp < Cfg::W_STA) {
    // ======================= prologue warps: rotation, operands, S -> S'
    const int pt = tid;
    const uint32_t lane_base = (uint32_t)(32 * (warp & 3)) << 16;
    const int k = pt % K2, g = pt / K2;  // rotation: pair k for the tokens of group g
    // dt and lam of token pt of a chunk (token Q: the next chunk's first),
    // loaded one chunk ahead as raw bf16 bits: converting them only where
    // they are used keeps the load latency behind a whole chunk of work
    const unsigned short* dt_bits = reinterpret_cast<const unsigned short*>(p.dt);
    const unsigned short* lam_bits = reinterpret_cast<const unsigned short*>(p.lam);
    // (token Q of the last chunk of a segment lies past its end: zero, the
    // carry takes the next token's previous-token term)
    // (with dt through softplus an absent token is marked kNoToken: its dt
    // must stay 0, not become softplus(bias))
    constexpr uint32_t kNoToken = 0xFFFFFFFFu;
    const bool dt_sp = (p.pro & M3_PRO_DT_SOFTPLUS) != 0;
    int pro_si = 0;  // the segment of the prologue's last chunk
    auto load_scalars = [&](int c, uint32_t& d, uint32_t& l, int tok) {
      d = dt_sp ? kNoToken : 0u;
      l = 0u;
      if (tok <= Q && c < nchunks) {
        const int si = seg_from(c, pro_si);
        const int64_t i = (int64_t)(c - sSegC0[si]) * Q + tok;
        if (i < seg_ntok(si)) {
          const int64_t row = (sSegTok0[si] + i) * H + seg_head(si);
          d = __ldg(dt_bits + row);
          l = lam_bits ? __ldg(lam_bits + row) : 0x3F80u;  // no lam: lam = 1
        }
      }
    };
    uint32_t d_cur, l_cur;
    load_scalars(0, d_cur, l_cur, pt);
    // prologue of chunk c: scalars, angle scan, rotation of B and C, X and W X.
    // Returns false when the pipeline was aborted.
    auto prologue = [&](int c, auto normtag) -> bool {
      constexpr bool NORM = decltype(normtag)::value;
      const int s = c % NS, xs = c % XB;  // stage, scalar slot
      uint8_t* stg = stage(s);
      const int si = seg_from(c, pro_si);
      pro_si = si;
      const float A = sSegA[si];
      // a segment starts from the phase 0 (its initial state is un-rotated);
      // these threads also wrote the previous chunk's phase
      const int pb = c & 1;  // this chunk's phase buffer
      if (c == sSegC0[si] && pt < K2) sPhi[pb][pt] = 0.f;
      uint32_t d_nxt, l_nxt;
      load_scalars(c + 1, d_nxt, l_nxt, pt);
      bool got = wait_or_abort(saddr(&bar_full[s]), (uint32_t)((c / NS) & 1), abort_flag);
      // scalar slot xs last served chunk c - XB: its output must be done
      if (got && c >= XB) got = wait_xfree(c - XB);
      // Every thread waited itself.  The vote on `got` is taken at the
      // chunk's closing barrier: a thread whose wait gave up computes on
      // whatever the tiles hold (no fault, no wait) and the group leaves
      // there together; one barrier fewer per chunk.
      if constexpr (NORM) {
        // ---- BC norm: 1 / rms of every B and C row (token, rank) of the tile
        //      as it landed; TPR adjacent threads per row, 16-byte chunks
        constexpr int TPR = NPRO / (2 * MR), CPT = N / 8 / TPR;
        const int row = pt / TPR, part = pt % TPR;
        const bool isC = row >= MR;
        const int rr = isC ? row - MR : row;
        const uint8_t* base = stg + (isC ? Cfg::OFF_C : Cfg::OFF_B);
        const uint32_t blk_bytes = isC ? (uint32_t)(MR * 128) : (uint32_t)Cfg::BB;
        float ss = 0.f;
        // (the state-only pass has no C tiles, and its stages no room for
        // them: the C rows' threads read nothing, and their sums are unused)
#pragma unroll
        for (int q = 0; q < CPT; ++q) {
          if (SO && isC) break;
          const int col = (part * CPT + q) * 8;
          const uint4 v = *reinterpret_cast<const uint4*>(base + (col / 64) * blk_bytes + sw128_offset(rr, col % 64));
          const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = bf2_to_f2(w4[e]);
            ss = fmaf(f.x, f.x, fmaf(f.y, f.y, ss));
          }
        }
#pragma unroll
        for (int o = TPR / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (part == 0) (isC ? sCScl : sBScl)[rr] = rsqrtf(ss * (1.f / N) + kBcNormEps);
      }
      // ---- per-token scalars and the inclusive scan of dt * A
      float dcur = __uint_as_float(d_cur << 16);
      const float lcur = __uint_as_float(l_cur << 16);
      if (dt_sp) dcur = d_cur == kNoToken ? 0.f : softplus_f(dcur + (p.dt_bias ? __ldg(p.dt_bias + seg_head(si)) : 0.f));
      if (pt <= Q) {
        sDt[pt] = dcur;
        sBet[pt] = (1.f - lcur) * dcur;
        if (pt < Q) sGam[xs][pt] = lcur * dcur;
      }
      // (whole warps take part in the shuffles: tokens Q..QW-1 contribute zero)
      constexpr int QW = (Q + 31) / 32 * 32;
      float v = (pt < Q) ? dcur * A : 0.f;
      if (pt < QW) {
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float u = __shfl_up_sync(0xffffffffu, v, o);
          if (lane >= o) v += u;
        }
        if (lane == 31) sWarpTot[warp] = v;
      }
      group_sync(1, NPRO);  // (also: sDt complete for the angle scan)
      if (pt < Q) {
        for (int w = 0; w < warp; ++w) v += sWarpTot[w];
        sLam[xs][pt] = v;
      }
      // ---- angle scan, part 1: per-group sums of dt * theta
      const __nv_bfloat16* th = reinterpret_cast<const __nv_bfloat16*>(stg + Cfg::OFF_TH);
      float om[TPG];
      if (!RE) {
        float part = 0.f;
#pragma unroll
        for (int ii = 0; ii < TPG; ++ii) {
          const int i = g * TPG + ii;
          om[ii] = sDt[i] * __bfloat162float(th[i * K2 + k]);
          part += om[ii];
        }
        sPsum[g][k] = part;
      }
      group_sync(1, NPRO);  // sLam and sPsum complete
      const float lam_end = sLam[xs][Q - 1];
      if constexpr (SO || xc_pro) {
        // ---- the state-only pass has no C to rotate and no scores: these
        //      warps also form W X as hi (over x) and lo (over theta, read
        //      above) parts for MMA 4, W_j = e^{Lam_end - Lam_j} (gamma_j +
        //      beta'_{j+1}), so that the stage's operands are ready with
        //      the prologue (and in the full pass, where they take this
        //      work, the f16 copy of X)
        uint8_t* Xs = stg + Cfg::OFF_X;
        uint8_t* WXlo = stg + Cfg::OFF_WXLO;
        uint8_t* Xb = xbuf(xs);
#pragma unroll 1
        for (int idx = pt; idx < MR * (P / 8); idx += NPRO) {
          const int row = idx / (P / 8), c8 = idx % (P / 8), j = row / R;
          const uint32_t o = sw128_offset(row, c8 * 8);
          const uint4 raw = *reinterpret_cast<const uint4*>(Xs + o);
          const float w = __expf(lam_end - sLam[xs][j]) * (sGam[xs][j] + sBet[j + 1]);
          const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t hx[4], hw[4], lw[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = bf2_to_f2(rw[q]);
            hx[q] = pack_half2(f.x, f.y);
            split_half2(w * f.x, w * f.y, hw[q], lw[q]);
          }
          if (!SO)
            *reinterpret_cast<uint4*>(Xb + sw128_offset(kperm(row), c8 * 8)) = make_uint4(hx[0], hx[1], hx[2], hx[3]);
          *reinterpret_cast<uint4*>(Xs + o) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(WXlo + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
      }
      if (pt < Q) {
        const float wp = sGam[xs][pt] + sBet[pt + 1];
        const float lt = sLam[xs][pt];
        sWp[xs][pt] = wp;
        sDw[xs][pt] = __expf(lam_end - lt) * wp;
        sBw[xs][pt] = __expf(-lt) * wp;
        sELam[xs][pt] = __expf(lt);
        if (pt == 0) sLamEnd[xs] = lam_end;
      }
      if (RE && g == 0) {  // theta = 0: the phase stays 0
        sPhiEndX[xs][k] = sPhi[pb][k];
        mbar_arrive_warp(saddr(&bar_phend[xs]));
      }
      // ---- angle scan, part 2, and the in-place rotation of B and C by
      //      e^{-i Phi_i}, Phi_i = phase at the chunk start + chunk-local sum
      if (RE) {  // theta = 0: B and C convert to f16 exactly, in place
        uint8_t* Bt = stg + Cfg::OFF_B;
        uint8_t* Ct = stg + Cfg::OFF_C;
        const int blk = (2 * k) / 64, col = (2 * k) % 64;
#pragma unroll
        for (int ii = 0; ii < TPG; ++ii) {
          const int i = g * TPG + ii;
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const uint32_t rc = sw128_offset(i * R + r, col);
            const uint32_t o = blk * (MR * 128) + rc, ob = blk * Cfg::BB + rc;
            // (both loads before the stores: the stores may alias them for the compiler)
            const float2 b = bf2_to_f2(*reinterpret_cast<const uint32_t*>(Bt + ob));
            const float2 cc = SO ? make_float2(0.f, 0.f) : bf2_to_f2(*reinterpret_cast<const uint32_t*>(Ct + o));
            *reinterpret_cast<uint32_t*>(Bt + ob) = pack_half2(b.x, b.y);
            if (!SO) *reinterpret_cast<uint32_t*>(Ct + o) = pack_half2(cc.x, cc.y);
          }
        }
      } else {
        float off = 0.f;
        float tot = 0.f;
#pragma unroll
        for (int gg = 0; gg < G; ++gg) {
          const float sv = sPsum[gg][k];
          off += (gg < g) ? sv : 0.f;
          tot += sv;
        }
        const float ph_end = sPhi[pb][k] + tot;
        uint8_t* Bt = stg + Cfg::OFF_B;
        uint8_t* Ct = stg + Cfg::OFF_C;
        uint8_t* Blo = stg + Cfg::OFF_BLO;
        uint8_t* Clo = stg + Cfg::OFF_CLO;
        const int blk = (2 * k) / 64, col = (2 * k) % 64;
        // angles of this thread's tokens, then all the sines and cosines,
        // then the rotations: independent work the scheduler can overlap
        float cs[TPG], sn[TPG];
        {
          float phi = sPhi[pb][k] + off;
#pragma unroll
          for (int ii = 0; ii < TPG; ++ii) {
            phi += om[ii];
            cs[ii] = -phi;
          }
#pragma unroll
          for (int ii = 0; ii < TPG; ++ii) sincos_reduced(cs[ii], &sn[ii], &cs[ii]);
        }
#pragma unroll
        for (int ii = 0; ii < TPG; ++ii) {
          const int i = g * TPG + ii;
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const uint32_t rc = sw128_offset(i * R + r, col);
            const uint32_t o = blk * (MR * 128) + rc, ob = blk * Cfg::BB + rc;
            // (both loads before the stores: the stores may alias them for
            // the compiler; the state-only pass has no C)
            float2 b = bf2_to_f2(*reinterpret_cast<const uint32_t*>(Bt + ob));
            float2 cc = SO ? make_float2(0.f, 0.f) : bf2_to_f2(*reinterpret_cast<const uint32_t*>(Ct + o));
            if constexpr (NORM) {
              const float fb = sBScl[i * R + r];
              b.x *= fb;
              b.y *= fb;
              if (!SO) {
                const float fc = sCScl[i * R + r];
                cc.x *= fc;
                cc.y *= fc;
              }
            }
            uint32_t hi, lo;
            split_half2(cs[ii] * b.x - sn[ii] * b.y, sn[ii] * b.x + cs[ii] * b.y, hi, lo);
            *reinterpret_cast<uint32_t*>(Bt + ob) = hi;
            *reinterpret_cast<uint32_t*>(Blo + ob) = lo;
            if (!SO) {
              split_half2(cs[ii] * cc.x - sn[ii] * cc.y, sn[ii] * cc.x + cs[ii] * cc.y, hi, lo);
              *reinterpret_cast<uint32_t*>(Ct + o) = hi;
              *reinterpret_cast<uint32_t*>(Clo + o) = lo;
            }
          }
        }
        if (g == 0) {  // the running phase after this chunk, reduced to [-pi, pi)
          sPhiEndX[xs][k] = fmaf(-rintf(ph_end * 0.15915494309189535f), 6.283185307179586f, ph_end);
          mbar_arrive_warp(saddr(&bar_phend[xs]));
        }
      }
      // the next chunk's running phase, in the other buffer (the same thread
      // wrote sPhiEndX); the closing barrier orders it, sDw and the last
      // reads of theta before the stage goes to the state warps and MMAs
      if (g == 0) sPhi[pb ^ 1][k] = sPhiEndX[xs][k];
      fence_async_smem();
      if (!group_and(1, NPRO, got)) return false;
      if (pt == 0) {
        mbar_arrive(saddr(&bar_opready[s]));
        if constexpr (xc_pro) mbar_arrive(saddr(&bar_xready[xs]));
      }
      d_cur = d_nxt;
      l_cur = l_nxt;
      return true;
    };
    // S -> S' of chunk c (after MMA 1 of c), in place in S[c & 1]: MMA 2 of
    // chunk c - 2, the last reader of that buffer's S', was issued before
    // MMA 1 of chunk c by the same thread
    auto scores = [&](int c) -> bool {
      const int s = c & 1, xs = c % XB;
      const float lam_end = sLamEnd[xs];
      // (a wait that gave up sets the CTA's abort flag: the next prologue's
      // vote sees it, and this step computes on whatever TMEM holds)
      wait_or_abort(saddr(&bar_sfull[s]), (uint32_t)((c >> 1) & 1), abort_flag);
      tc_fence_after();
      // warp w covers accumulator rows 16(w%4) .. +15 (TMEM lane quarter w%4)
      // and one slice of CPH columns; with the 16x256b shape thread `lane`
      // holds rows r0 = 16(w%4) + lane/4 and r0 + 8, columns 8g + 2(lane%4)
      // + {0, 1} of each 8-column group g: all 32 lanes carry data
      const int q4 = warp & 3;
      const int r0 = 16 * q4 + lane / 4;
      const int it0 = r0 / R, it1 = (r0 + 8) / R;
      // last token held by this warp's rows: column blocks past it are all masked
      const int it_warp = (16 * q4 + 15) / R;
      const float elam0 = sELam[xs][it0], lam0 = sLam[xs][it0], gam0 = sGam[xs][it0];
      const float elam1 = sELam[xs][it1], lam1 = sLam[xs][it1], gam1 = sGam[xs][it1];
      const bool factor = lam_end > -60.f;  // e^{Lam_t} and e^{-Lam_j} both stay normal floats
      constexpr int CPH = MR / (NPRO / 128);  // columns per warp (warps w, w+4, ... share rows)
      const int cbeg = (warp >> 2) * CPH;
      const int cl = 2 * (lane % 4);        // this thread's column pair inside each 8-column group
#pragma unroll 1
      for (int cb = 0; cb < CPH; cb += 16) {
        const uint32_t ta = tmem + lane_base + Cfg::COL_S + s * MR + cbeg + cb;
        // the block's S' as 8 columns of hi words, then 8 of lo words; the
        // word of columns (8 gg + cl, +1) of each row goes to word column
        // cl + gg (the 16x256b store puts this thread's registers 2i, 2i + 1
        // of each group at word columns cl, cl + 1), which is the order kperm
        // describes
        uint32_t wv[8];  // [hi, lo][(r0, gg 0), (r0, gg 1), (r0 + 8, gg 0), (r0 + 8, gg 1)]
        if ((cbeg + cb) / R > it_warp) {  // all masked: zeros
#pragma unroll
          for (int i = 0; i < 8; ++i) wv[i] = 0u;
        } else {
          float sv[8];  // [group gg][4]: (r0, c), (r0, c+1), (r0+8, c), (r0+8, c+1)
          tmem_ld16x256b_x2(ta, sv);
          tmem_ld_wait();
#pragma unroll
          for (int gg = 0; gg < 2; ++gg) {
            const int j = cbeg + cb + 8 * gg + cl;  // first of this thread's two columns
            float bw2[2];
            if (R == 1) {
              const float2 w2 = *reinterpret_cast<const float2*>(&sBw[xs][j]);
              bw2[0] = w2.x;
              bw2[1] = w2.y;
            } else {
              bw2[0] = sBw[xs][j / R];
              bw2[1] = sBw[xs][(j + 1) / R];
            }
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              const int it = rr ? it1 : it0;
              const float elam_t = rr ? elam1 : elam0, lam_t = rr ? lam1 : lam0, gam_t = rr ? gam1 : gam0;
              float e[2];
#pragma unroll
              for (int u = 0; u < 2; ++u) {
                const int jt = (j + u) / R;
                const float sij = sv[4 * gg + 2 * rr + u];
                const float off = factor ? sij * bw2[u] * elam_t : sij * __expf(lam_t - sLam[xs][jt]) * sWp[xs][jt];
                e[u] = jt < it ? off : (jt == it ? sij * gam_t : 0.f);
              }
              split_half2(e[0], e[1], wv[2 * rr + gg], wv[4 + 2 * rr + gg]);
            }
          }
        }
        tmem_st16x256b_x2(ta, wv);
      }
      // each warp signals its own columns to MMA 2: no barrier of the group
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive_warp(saddr(&bar_spready[s]));
      return true;
    };
    // the prologue runs one chunk ahead of S -> S', which waits for MMA 1
    // compiled once with and once without the BC norm (the real-state
    // variant has none: its B and C reach the MMAs without a lo part)
    auto run = [&](auto normtag) {
      bool alive = prologue(0, normtag);
      for (int c = 0; c < nchunks && alive; ++c) {
        if (c + 1 < nchunks && !prologue(c + 1, normtag)) break;
        if (!SO) alive = scores(c);
      }
    };
    if (!RE && (p.pro & M3_PRO_BC_NORM))
      run(BoolTag<true>{});
    else
      run(BoolTag<false>{});
  } else if (warp < Cfg::W_MMA) {
    // ======================= state warps: state step and output epilogue
    const int tt = tid - NPRO;
    const int q4 = warp & 3;
    const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
    const int g_row = acc_row_of(N, q4, lane);  // state row owned by this thread (-1: none)
    // initial state of segment si: h'_{-1} = h0 + beta'_0 * sum_r Bprev_r
    // xprev_r^T (realified rows), h0 and the carry from the caller's state
    // (zero without one) or from a handover slot, whose writer publishes it
    // with a release store of its flag; also R = f16(G') for the first MMA 3
    // of the segment.
    // product of the segment's chunk decays (the state-only pass reports it)
    float seg_decay = 1.f;
    auto init_seg = [&](int si) -> bool {
      const int4 sg = sSeg[si];
      seg_decay = 1.f;
      const int unit = sg.x, head = unit % H;
      const bool from_slot = (sg.w & SEG_SRC_SLOT) != 0;
      const bool split = (sg.w & SEG_SPLIT) != 0;
      const int slot = sg.w >> 8;
      // the first token's dt and lam, loaded before the wait below (their
      // latency overlaps it)
      const int64_t row0 = sSegTok0[si] * H + head;
      const __nv_bfloat16 dt0_raw = p.dt[row0];
      const __nv_bfloat16 lm0_raw = p.lam ? p.lam[row0] : __float2bfloat16(1.f);  // no lam: lam = 1
      if (from_slot && !split) {  // bounded wait for the CTA that runs the first part of this unit
        bool ok = false;
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t i = 0; i < kMaxPolls; ++i) {
          int f;
          asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(f) : "l"(p.xflag + slot) : "memory");
          if (f) {
            ok = true;
            break;
          }
          if ((i & 63u) == 0 && (abort_flag->flag || globaltimer_ns() - t0 > abort_flag->limit_ns)) break;
        }
        if (!group_and(2, NSTA, ok)) {
          if (tt == 0) {
            abort_flag->flag = 1;
            atomicExch(&g_status, (int)M3_ERR_TIMEOUT);
          }
          return false;
        }
      }
      // (the state-only pass starts every piece from the zero state)
      const float* h0 = SO ? nullptr
                           : from_slot ? p.xh + (int64_t)slot * K2 * P * 2
                                       : (p.h ? p.h + (int64_t)unit * K2 * P * 2 : nullptr);
      const __nv_bfloat16* cB = from_slot ? p.xB + (int64_t)slot * R * N : (p.prev_B ? p.prev_B + (int64_t)unit * R * N : nullptr);
      const __nv_bfloat16* cx = from_slot ? p.xx + (int64_t)slot * R * P : (p.prev_x ? p.prev_x + (int64_t)unit * R * P : nullptr);
      if (split) {  // the previous token's rows, or the caller's carry at the unit's start
        const int64_t tp = sSegTok0[si] - 1;
        if (sg.y > 0) {
          cB = p.B + (tp * p.G + head / (H / p.G)) * R * N;
          cx = p.x + (tp * H + head) * R * P;
        } else {
          cB = p.prev_B ? (SO ? p.prev_B + (int64_t)unit * R * N : p.xB + (int64_t)slot * R * N) : nullptr;
          cx = p.prev_x ? (SO ? p.prev_x + (int64_t)unit * R * P : p.xx + (int64_t)slot * R * P) : nullptr;
        }
      }
      const float dt0 = scan_dt(__bfloat162float(dt0_raw), p.pro, p.dt_bias, head);
      const float lm0 = __bfloat162float(lm0_raw);
      const float bet0 = (1.f - lm0) * dt0;
      const bool norm_c = (p.pro & M3_PRO_BC_NORM) && cB;  // BC norm of the carried B rows
      if (norm_c) {
        for (int r = tt >> 5; r < R; r += NSTA / 32) {
          const float sc = warp_rms_scale(cB + r * N, N, tt & 31);
          if ((tt & 31) == 0) sCarryScl[r] = sc;
        }
      }
      // the carry's B entries of this thread's row (scaled by beta'_0) and
      // the carried x rows (into shared memory): read once, not per column
      // block, so that the column loop waits only on the state's loads
      float cbr[R];
      if (cB) {
        for (int i = tt; i < R * P; i += NSTA) sCarryX[i] = cx[i];
#pragma unroll
        for (int r = 0; r < R; ++r) cbr[r] = g_row >= 0 ? __bfloat162float(cB[r * N + g_row]) : 0.f;
      }
      if (norm_c || cB) group_sync(2, NSTA);
      if (cB) {
#pragma unroll
        for (int r = 0; r < R; ++r) cbr[r] *= bet0 * (norm_c ? sCarryScl[r] : 1.f);
      }
      // the 16 columns of pair g_row / 2 are 128 contiguous bytes (re, im
      // interleaved): the re lane loads columns cb..cb+7, the im lane
      // cb+8..cb+15, and each passes the other the half it needs; the next
      // block's loads are issued before this block's are used
      const bool re = (g_row & 1) == 0;
      auto load_own = [&](int cb, float (&o)[16]) {
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] = 0.f;
        if (h0 && g_row >= 0) {
          const float4* hs = reinterpret_cast<const float4*>(h0 + (int64_t)(g_row >> 1) * P * 2 + (cb + (re ? 0 : 8)) * 2);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float4 f = hs[q];
            o[4 * q] = f.x;
            o[4 * q + 1] = f.y;
            o[4 * q + 2] = f.z;
            o[4 * q + 3] = f.w;
          }
        }
      };
      float nxt[16];
      load_own(0, nxt);
      for (int cb = 0; cb < P; cb += 16) {
        float v[16], own[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          v[i] = 0.f;
          own[i] = nxt[i];
        }
        if (cb + 16 < P) load_own(cb + 16, nxt);
        if (h0) {
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            // (selects, not lane-dependent indices, keep the arrays in registers)
            const float mine = re ? own[2 * i] : own[2 * i + 1];  // this lane's part of its own columns
            const float other = __shfl_xor_sync(0xffffffffu, re ? own[2 * i + 1] : own[2 * i], 1);
            v[i] = re ? mine : other;
            v[8 + i] = re ? other : mine;
          }
        }
        if (g_row >= 0 && cB) {
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const __nv_bfloat16* xp = sCarryX + r * P + cb;
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = fmaf(cbr[r], __bfloat162float(xp[i]), v[i]);
          }
        }
        tmem_st16(tmem + lane_base + Cfg::COL_G + cb, v);
        if (!SO && g_row >= 0) {  // R = f16(G') for MMA 3 of the segment's first chunk
#pragma unroll
          for (int pc = 0; pc < 16; pc += 8)
            *reinterpret_cast<uint4*>(Rt + sw128_offset(g_row, cb + pc)) =
                make_uint4(pack_half2(v[pc], v[pc + 1]), pack_half2(v[pc + 2], v[pc + 3]),
                           pack_half2(v[pc + 4], v[pc + 5]), pack_half2(v[pc + 6], v[pc + 7]));
        }
      }
      tmem_st_wait();
      fence_async_smem();
      tc_fence_before();
      group_sync(2, NSTA);
      if (!SO && tt == 0) mbar_arrive(saddr(&bar_stready));
      // the next segment's initial state, when it is the caller's: into L2
      // now, so that its loads hit there when that segment starts
      if (si + 1 < nseg && !(sSeg[si + 1].w & SEG_SRC_SLOT) && p.h) {
        const char* nh = reinterpret_cast<const char*>(p.h + (int64_t)sSeg[si + 1].x * K2 * P * 2);
        for (int off = tt * 128; off < K2 * P * 2 * 4; off += NSTA * 128)
          asm volatile("prefetch.global.L2 [%0];" ::"l"(nh + off));
      }
      return true;
    };
    // final state of segment si (h of its last token, rotated back by the
    // phase after its last chunk c) and carry (that token's B and x), to the
    // caller's state or to a handover slot (then published with a release
    // store of the slot's flag)
    // (the state-only pass: the segment's own final state to seg_h and its
    // decay and rotation e^{Lam + i Phi} to seg_alpha, then the release of
    // the last chunk's scalar slot; a segment that a later one continues in
    // a split schedule writes nothing)
    auto finalize = [&](int si, int c) -> bool {
      const int4 sg = sSeg[si];
      const int unit = sg.x, head = unit % H;
      if (!SO && (sg.w & SEG_NO_FINAL)) return true;
      const bool to_slot = !SO && (sg.w & SEG_DST_SLOT) != 0;
      const int slot = sg.w >> 8;
      float* hd = SO ? p.seg_h + (int64_t)slot * K2 * P * 2
                     : (to_slot ? p.xh + (int64_t)slot * K2 * P * 2 : (p.h ? p.h + (int64_t)unit * K2 * P * 2 : nullptr));
      __nv_bfloat16* cB = SO ? nullptr : to_slot ? p.xB + (int64_t)slot * R * N : (p.prev_B ? p.prev_B + (int64_t)unit * R * N : nullptr);
      __nv_bfloat16* cx = SO ? nullptr : to_slot ? p.xx + (int64_t)slot * R * P : (p.prev_x ? p.prev_x + (int64_t)unit * R * P : nullptr);
      if (hd) {  // h = e^{i Phi_end} G' (pairs of rows are (re, im) in adjacent lanes)
        // the prologue of chunk c + XB (the slot's next writer) needs the
        // output of chunk c, which follows: this parity wait cannot fall behind
        // (a group vote: every state thread leaves together, or none does)
        if (!group_and(2, NSTA, wait_or_abort(saddr(&bar_phend[c % XB]), (uint32_t)((c / XB) & 1), abort_flag)))
          return false;
        float cs = 1.f, sn = 0.f;
        if (g_row >= 0) sincosf(sPhiEndX[c % XB][g_row >> 1], &sn, &cs);
        const bool re = (g_row & 1) == 0;
        if (SO && g_row >= 0 && re)
          p.seg_alpha[(int64_t)slot * K2 + (g_row >> 1)] = make_float2(seg_decay * cs, seg_decay * sn);
        for (int cb = 0; cb < P; cb += 16) {
          float v[16];
          tmem_ld16(tmem + lane_base + Cfg::COL_G + cb, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float other = __shfl_xor_sync(0xffffffffu, v[i], 1);
            v[i] = re ? (cs * v[i] - sn * other) : (sn * other + cs * v[i]);
          }
          // (re, im) of columns cb..cb+7 from the re lane, cb+8..cb+15 from
          // the im lane: 64 contiguous bytes each
          float out[16];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float other = __shfl_xor_sync(0xffffffffu, re ? v[8 + i] : v[i], 1);
            out[2 * i] = re ? v[i] : other;
            out[2 * i + 1] = re ? other : v[8 + i];
          }
          if (g_row >= 0) {
            float4* hs = reinterpret_cast<float4*>(hd + (int64_t)(g_row >> 1) * P * 2 + (cb + (re ? 0 : 8)) * 2);
#pragma unroll
            for (int q = 0; q < 4; ++q) hs[q] = make_float4(out[4 * q], out[4 * q + 1], out[4 * q + 2], out[4 * q + 3]);
          }
        }
      }
      if (cB) {
        const int64_t last = (sSegTok0[si] + seg_ntok(si) - 1) * H + head;
        const int64_t lastg = (sSegTok0[si] + seg_ntok(si) - 1) * p.G + head / (H / p.G);
        for (int i = tt; i < R * N; i += NSTA) cB[i] = p.B[lastg * R * N + i];
        for (int i = tt; i < R * P; i += NSTA) cx[i] = p.x[last * R * P + i];
      }
      if (to_slot) {
        __threadfence();
        group_sync(2, NSTA);
        if (tt == 0 && p.fault != M3_TEST_FAULT_SKIP_HANDOVER_RELEASE)
          asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p.xflag + slot), "r"(1) : "memory");
      }
      if (SO) {  // the last chunk's scalars (its phase) are read: release the slot
        group_sync(2, NSTA);
        if (tt == 0) mbar_arrive(saddr(&bar_xfree[c % XB]));
      }
      return true;
    };
    // X of chunk c to f16 (slot c % XB) and W X as hi (over x) and lo (over
    // theta, or its own area) parts: after the prologue of chunk c (its
    // weights, and its last read of theta)
    auto xconv = [&](int c) -> bool {
      const int s = c % NS, xs = c % XB;
      uint8_t* stg = stage(s);
      bool got = wait_or_abort(saddr(&bar_opready[s]), (uint32_t)((c / NS) & 1), abort_flag);
      if (!SO && got && c >= XB) got = wait_xfree(c - XB);  // (SO: no X slot)
      if (!group_and(2, NSTA, got)) return false;
      {
        uint8_t* Xs = stg + Cfg::OFF_X;
        uint8_t* WXlo = stg + Cfg::OFF_WXLO;
        uint8_t* Xb = xbuf(xs);
#pragma unroll 2
        for (int idx = tt; idx < MR * (P / 8); idx += NSTA) {
          const int row = idx / (P / 8), c8 = idx % (P / 8);
          const uint32_t o = sw128_offset(row, c8 * 8);
          const uint4 raw = *reinterpret_cast<const uint4*>(Xs + o);
          const float w = sDw[xs][row / R];
          const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
          uint32_t hx[4], hw[4], lw[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = bf2_to_f2(rw[q]);
            hx[q] = pack_half2(f.x, f.y);
            split_half2(w * f.x, w * f.y, hw[q], lw[q]);
          }
          if (!SO)
            *reinterpret_cast<uint4*>(Xb + sw128_offset(kperm(row), c8 * 8)) = make_uint4(hx[0], hx[1], hx[2], hx[3]);
          *reinterpret_cast<uint4*>(Xs + o) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
          *reinterpret_cast<uint4*>(WXlo + o) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
        }
        fence_async_smem();
        group_sync(2, NSTA);
        if (tt == 0) mbar_arrive(saddr(&bar_xready[xs]));
      }
      return true;
    };
    // state step of chunk c, in the rotating frame: G' <- e^{Lam_end} G' + S_c
    // (S_c from MMA 4 of chunk c), then R = f16(G') for MMA 3 of chunk c + 1
    // once MMA 3 of chunk c has read the previous R.  After the last chunk of
    // a segment the next segment's initial state provides that R instead.
    auto state = [&](int c) -> bool {
      const int xs = c % XB;
      const bool pub = !seg_last(c);
      const int sb = SO ? (c & 1) : 0;  // chunk-local state buffer
      const uint32_t col_sc = sb ? Cfg::COL_SC1 : Cfg::COL_SC;
      bool got = wait_or_abort(saddr(&bar_scfull[sb]), (uint32_t)((SO ? c >> 1 : c) & 1), abort_flag);
      if (!SO && got) got = wait_or_abort(saddr(&bar_rfree), (uint32_t)(c & 1), abort_flag);
      if (!group_and(2, NSTA, got)) return false;
      tc_fence_after();
      const float elam_end = __expf(sLamEnd[xs]);
      seg_decay *= elam_end;
#pragma unroll 1
      for (int hc = 0; hc < P; hc += 16) {
        float g[16], sc[16];
        tmem_ld16(tmem + lane_base + Cfg::COL_G + hc, g);
        tmem_ld16(tmem + lane_base + col_sc + hc, sc);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) g[i] = fmaf(elam_end, g[i], sc[i]);
        tmem_st16(tmem + lane_base + Cfg::COL_G + hc, g);
        if (!SO && pub && g_row >= 0) {
#pragma unroll
          for (int pc = 0; pc < 16; pc += 8)
            *reinterpret_cast<uint4*>(Rt + sw128_offset(g_row, hc + pc)) =
                make_uint4(pack_half2(g[pc], g[pc + 1]), pack_half2(g[pc + 2], g[pc + 3]),
                           pack_half2(g[pc + 4], g[pc + 5]), pack_half2(g[pc + 6], g[pc + 7]));
        }
      }
      tmem_st_wait();
      fence_async_smem();
      tc_fence_before();
      group_sync(2, NSTA);
      if (tt == 0) {
        if (!SO && pub) mbar_arrive(saddr(&bar_stready));
        mbar_arrive(saddr(&bar_scfree[sb]));
        // the state-only pass releases the chunk's scalar slot here (the
        // segment's last chunk: after finalize has read its phase)
        if (SO && pub) mbar_arrive(saddr(&bar_xfree[xs]));
      }
      return true;
    };

    // output of chunk c: y = Y + e^{Lam_t} Yi + D x, needs MMAs 2 and 3 of chunk c
    auto output = [&](int c, auto ybf) -> bool {
      const int s = c & 1, xs = c % XB;
      const int si = seg_of(c), head = seg_head(si);
      const int64_t cc = c - sSegC0[si];
      const int64_t ct0 = sSegTok0[si] + cc * Q;
      const int64_t left = seg_ntok(si) - cc * Q;
      const int nvalid = left < Q ? (int)left : Q;
      const float Dh = sSegD[si];
      if (!group_and(2, NSTA, wait_or_abort(saddr(&bar_yfull[s]), (uint32_t)((c >> 1) & 1), abort_flag)))
        return false;
      tc_fence_after();
      const uint8_t* Xb = xbuf(xs);
      // 16x256b shape: thread `lane` holds rows r0 = 16(w%4) + lane/4 and
      // r0 + 8, columns 8g + 2(lane%4) + {0, 1} of each 8-column group g, so
      // every store of a warp fills eight whole 32-byte sectors of y
      const int r0 = 16 * q4 + lane / 4, cl = 2 * (lane % 4);
      bool valid[2];
      float el[2];
      int64_t yrow[2];
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int t = r0 + 8 * rr, it = t / R, rk = t % R;
        valid[rr] = it < nvalid;
        el[rr] = sELam[xs][it];
        yrow[rr] = ((ct0 + it) * H + head) * (R * P) + rk * P;
      }
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        float a[16], b[16];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          float ta[8], tb[8];
          tmem_ld16x256b_x2(tmem + lane_base + Cfg::COL_Y + s * P + 32 * half + 16 * q, ta);
          tmem_ld16x256b_x2(tmem + lane_base + Cfg::COL_YI + s * P + 32 * half + 16 * q, tb);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            a[8 * q + i] = ta[i];
            b[8 * q + i] = tb[i];
          }
        }
        tmem_ld_wait();
#pragma unroll
        for (int g8 = 0; g8 < 4; ++g8) {
          const int col = 32 * half + 8 * g8 + cl;
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const uint32_t xv = *reinterpret_cast<const uint32_t*>(Xb + sw128_offset(kperm(r0 + 8 * rr), col));
            const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&xv));
            const int i0 = 4 * g8 + 2 * rr;
            const float o0 = fmaf(Dh, f.x, fmaf(el[rr], b[i0], a[i0]));
            const float o1 = fmaf(Dh, f.y, fmaf(el[rr], b[i0 + 1], a[i0 + 1]));
            if (valid[rr]) st_y2(p.y, yrow[rr] + col, o0, o1, decltype(ybf)::value);
          }
        }
      }
      tc_fence_before();
      group_sync(2, NSTA);
      if (tt == 0) mbar_arrive(saddr(&bar_xfree[xs]));
      return true;
    };
    // order, chunk n after chunk: X of chunk n (unless XC) after its prologue,
    // the output of chunk n - 1 (after its MMAs 2 and 3), then the
    // state step of chunk n (its R is needed by the next MMA 3 long before
    // the stage is released).  A segment's initial state is loaded before
    // its first chunk and its final state written after its last, outside
    // the per-chunk loop, whose code stays small and contiguous (the roles
    // of one SM share its instruction cache).  `alive` is the same in every
    // state warp: each step ends in a group vote.
    // The loop is compiled once per output type (y f32 or bf16), so that the
    // store needs no branch in the chunk loop.
    auto run = [&](auto ybf) {
      bool alive = true;
      int n = 0;
      for (int si = 0; si < nseg && alive; ++si) {
        if (!init_seg(si)) break;
        const int end = sSegC0[si + 1];
        for (; n < end; ++n) {
          if ((!SO && !xc_pro && !xconv(n)) || (!SO && n >= 1 && !output(n - 1, ybf)) || !state(n)) {
            alive = false;
            break;
          }
        }
        if (alive) alive = finalize(si, n - 1);
      }
      if (!SO && alive) output(nchunks - 1, ybf);
    };
    if (p.ybf)
      run(BoolTag<true>{});
    else
      run(BoolTag<false>{});
  } else if (warp == Cfg::W_MMA || warp == Cfg::W_MMA2) {
    // ======================= MMA warps (one thread each issues)
    // K-major operand tiles: 16-element K step = 32 B inside a 128 B row, 64-column blocks MR*128 B apart
    auto kmaj = [](uint32_t base, int ks, uint32_t block_bytes) {
      return smem_desc(base + (ks / 4) * block_bytes + (ks % 4) * 32, 16, 1024, kSwizzle128B);
    };
    // MN-major operand tiles: 16-element K step = two 8-row atoms
    auto mnmaj = [](uint32_t base, int ks, uint32_t lbo) {
      return smem_desc(base + ks * 2048, lbo, 1024, kSwizzle128B);
    };
    if (lane == 0 && warp == Cfg::W_MMA && !SO) {  // (the state-only pass has no intra-chunk products)
      // intra-chunk products, MMA 1 one chunk ahead of MMA 2
      auto mma1 = [&](int c) -> bool {
        const int s = c & 1, sg = c % NS;  // S buffer, stage
        uint8_t* stg = stage(sg);
        const uint32_t Ct = saddr(stg + Cfg::OFF_C), Bt = saddr(stg + Cfg::OFF_B);
        const uint32_t Clo = saddr(stg + Cfg::OFF_CLO), Blo = saddr(stg + Cfg::OFF_BLO);
        if (!wait_or_abort(saddr(&bar_opready[sg]), (uint32_t)((c / NS) & 1), abort_flag)) return false;
        // S[s] last held the S' of chunk c - 2: MMA 2 of that chunk, issued
        // before this by this thread, read it (tcgen05 MMAs of one thread run
        // in issue order), after S -> S' of chunk c - 2 was done
        tc_fence_after();
        // S = C B^T = Chi Bhi^T + Chi Blo^T + Clo Bhi^T   (M = MR, N = MR, K = N)
        constexpr uint32_t idesc = idesc_f16_f32(MR, MR, 0, 0);
        const uint32_t d = tmem + Cfg::COL_S + s * MR;
#pragma unroll 1
        for (int ks = 0; ks < N / 16; ++ks) {
          mma_f16(d, kmaj(Ct, ks, MR * 128), kmaj(Bt, ks, Cfg::BB), idesc, ks > 0);
          if (!RE) {  // the lo parts of the rotated operands
            mma_f16(d, kmaj(Ct, ks, MR * 128), kmaj(Blo, ks, Cfg::BB), idesc, 1);
            mma_f16(d, kmaj(Clo, ks, MR * 128), kmaj(Bt, ks, Cfg::BB), idesc, 1);
          }
        }
        mma_commit(saddr(&bar_sfull[s]));
        mma_commit(saddr(&bar_free[sg]));
        return true;
      };
      // intra-chunk products, MMA 1 one chunk ahead of MMA 2
      bool alive = mma1(0);
      for (int c = 0; c < nchunks && alive; ++c) {
        const int s = c & 1;
        if (c + 1 < nchunks && !mma1(c + 1)) break;
        if (!wait_or_abort(saddr(&bar_spready[s]), (uint32_t)((c >> 1) & 1), abort_flag)) break;
        if (!wait_or_abort(saddr(&bar_xready[c % XB]), (uint32_t)((c / XB) & 1), abort_flag)) break;  // X of chunk c
        if (c >= 2 && !wait_xfree(c - 2)) break;  // Y[s] last held the output of chunk c - 2
        tc_fence_after();
        // Y[s] = S' X = S'hi X + S'lo X   (M = MR, N = P, K = MR; X is exact in f16):
        // S' from TMEM (K step ks: 8 columns of hi words at 16 ks, then 8 of lo)
        const uint32_t Xb = saddr(xbuf(c % XB));
        const uint32_t sp = tmem + Cfg::COL_S + s * MR;
        constexpr uint32_t idesc = idesc_f16_f32(MR, P, 0, 1);
#pragma unroll 1
        for (int ks = 0; ks < MR / 16; ++ks) {
          mma_f16_ta(tmem + Cfg::COL_Y + s * P, sp + 16 * ks, mnmaj(Xb, ks, MR * 128), idesc, ks > 0);
          mma_f16_ta(tmem + Cfg::COL_Y + s * P, sp + 16 * ks + 8, mnmaj(Xb, ks, MR * 128), idesc, 1);
        }
        mma_commit(saddr(&bar_yfull[s]));
        mma_commit(saddr(&bar_xfree[c % XB]));
      }
      // on every exit, normal or aborted: no product still writes TMEM when it is freed
      mma_commit(saddr(&bar_mdone[0]));
      mbar_wait(saddr(&bar_mdone[0]), 0, kMaxPolls);
    } else if (lane == 0 && warp == Cfg::W_MMA2) {
      // MMA 3 (inter-chunk output) and MMA 4 (chunk-local state) of chunk c.
      // MMA 3 needs only this chunk's C and the R of the previous state step,
      // so it goes first; the stage is released when MMA 4 is done.
      for (int c = 0; c < nchunks; ++c) {
        const int s = c & 1, sg = c % NS;  // Yi buffer, stage
        uint8_t* stg = stage(sg);
        const uint32_t Ct = saddr(stg + Cfg::OFF_C), Bt = saddr(stg + Cfg::OFF_B);
        const uint32_t Clo = saddr(stg + Cfg::OFF_CLO), Blo = saddr(stg + Cfg::OFF_BLO);
        const uint32_t WXt = saddr(stg + Cfg::OFF_X), WXlo = saddr(stg + Cfg::OFF_WXLO);
        // C of the stage rotated (prologue); R of the state at the start of chunk c
        // written; Yi[s] free (output of chunk c - 2 done)
        if (!wait_or_abort(saddr(&bar_opready[sg]), (uint32_t)((c / NS) & 1), abort_flag)) break;
        if (!SO) {
          if (!wait_or_abort(saddr(&bar_stready), (uint32_t)(c & 1), abort_flag)) break;
          if (c >= 2 && !wait_xfree(c - 2)) break;
          tc_fence_after();
          {  // Yi[s] = C R = Chi R + Clo R   (M = MR, N = P, K = N)
            constexpr uint32_t idesc = idesc_f16_f32(MR, P, 0, 1);
#pragma unroll 1
            for (int ks = 0; ks < N / 16; ++ks) {
              mma_f16(tmem + Cfg::COL_YI + s * P, kmaj(Ct, ks, MR * 128), mnmaj(saddr(Rt), ks, N * 128), idesc, ks > 0);
              if (!RE)
                mma_f16(tmem + Cfg::COL_YI + s * P, kmaj(Clo, ks, MR * 128), mnmaj(saddr(Rt), ks, N * 128), idesc, 1);
            }
          }
          mma_commit(saddr(&bar_rfree));
          mma_commit(saddr(&bar_yfull[s]));
        }
        // W X converted (state warps; XC and SO: the prologue, with the
        // operands); the buffer's previous chunk-local state folded into the
        // state (S_{c-1}; SO: S_{c-2})
        if (!SO && !wait_or_abort(saddr(&bar_xready[c % XB]), (uint32_t)((c / XB) & 1), abort_flag)) break;
        const int sb = SO ? (c & 1) : 0;
        const uint32_t col_sc = sb ? Cfg::COL_SC1 : Cfg::COL_SC;
        if (SO ? (c >= 2 && !wait_or_abort(saddr(&bar_scfree[sb]), (uint32_t)(((c >> 1) - 1) & 1), abort_flag))
               : (c >= 1 && !wait_or_abort(saddr(&bar_scfree[0]), (uint32_t)((c - 1) & 1), abort_flag)))
          break;
        tc_fence_after();
        {  // S_c = B^T (W X) = Bhi^T WXhi + Bhi^T WXlo + Blo^T WXhi   (M = N, N = P, K = MR)
          constexpr uint32_t idesc = idesc_f16_f32(N, P, 1, 1);
#pragma unroll 1
          for (int ks = 0; ks < MR / 16; ++ks) {
            mma_f16(tmem + col_sc, mnmaj(Bt, ks, Cfg::BB), mnmaj(WXt, ks, MR * 128), idesc, ks > 0);
            mma_f16(tmem + col_sc, mnmaj(Bt, ks, Cfg::BB), mnmaj(WXlo, ks, MR * 128), idesc, 1);
            if (!RE) mma_f16(tmem + col_sc, mnmaj(Blo, ks, Cfg::BB), mnmaj(WXt, ks, MR * 128), idesc, 1);
          }
        }
        // each commit tracks every product issued so far by this thread
        mma_commit(saddr(&bar_scfull[sb]));
        mma_commit(saddr(&bar_free[sg]));
      }
      mma_commit(saddr(&bar_mdone[1]));
      mbar_wait(saddr(&bar_mdone[1]), 0, kMaxPolls);
    }
  } else {
    // ======================= TMA warp (one thread issues)
    if (lane == 0) {
      int issued[3] = {0, 0, 0};
      const int hpg = H / p.G;  // heads per B / C group
      auto issue = [&](int c) {
        const int s = c % NS;
        uint8_t* stg = stage(s);
        const uint32_t bar = saddr(&bar_full[s]);
        const int si = seg_of(c), head = seg_head(si);
        const int t = (int)(sSegTok0[si] + (int64_t)(c - sSegC0[si]) * Q);
        mbar_arrive_expect_tx(bar, SO ? Cfg::STAGE_TX - Cfg::CT_BYTES : Cfg::STAGE_TX);  // (SO: no C tile)
        tma_load_4d(saddr(stg + Cfg::OFF_X), &tm_x, bar, 0, 0, head, t);
#pragma unroll
        for (int kb = 0; kb < N / 64; ++kb) {
          tma_load_4d(saddr(stg + Cfg::OFF_B + kb * Cfg::BB), &tm_B, bar, 64 * kb, 0, head / hpg, t);
          if (!SO) tma_load_4d(saddr(stg + Cfg::OFF_C + kb * MR * 128), &tm_C, bar, 64 * kb, 0, head / hpg, t);
        }
        if (!RE) tma_load_3d(saddr(stg + Cfg::OFF_TH), &tm_th, bar, 0, head, t);
        ++issued[s];
      };
      // the stage of chunk c + NS frees only when chunk c is done; the chunk
      // after it is fetched into L2 meanwhile, so its load then hits in L2
      auto prefetch = [&](int c) {
        if (c >= nchunks) return;
        const int si = seg_of(c), head = seg_head(si);
        const int t = (int)(sSegTok0[si] + (int64_t)(c - sSegC0[si]) * Q);
        tma_prefetch_4d(&tm_x, 0, 0, head, t);
#pragma unroll
        for (int kb = 0; kb < N / 64; ++kb) {
          tma_prefetch_4d(&tm_B, 64 * kb, 0, head / hpg, t);
          if (!SO) tma_prefetch_4d(&tm_C, 64 * kb, 0, head / hpg, t);
        }
        if (!RE) tma_prefetch_3d(&tm_th, 0, head, t);
      };
      tma_prefetch_desc(&tm_x);
      tma_prefetch_desc(&tm_B);
      if (!SO) tma_prefetch_desc(&tm_C);
      if (!RE) tma_prefetch_desc(&tm_th);
      for (int c = 0; c < NS && c < nchunks; ++c) issue(c);
      prefetch(NS);
      for (int c = 0; c + NS < nchunks; ++c) {
        if (!wait_or_abort(saddr(&bar_free[c % NS]), (uint32_t)((c / NS) & 1), abort_flag)) break;
        issue(c + NS);
        prefetch(c + NS + 1);
      }
      // every load issued must have landed before the CTA's shared memory goes away
      for (int s = 0; s < NS; ++s)
        if (issued[s] > 0) mbar_wait(saddr(&bar_full[s]), (uint32_t)((issued[s] - 1) & 1), kMaxPolls);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, Cfg::TMEM_COLS);
}

// ------------------------------------------------------------------ host side

typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline PFN_encodeTiled get_encode_tiled() {
  static PFN_encodeTiled fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_encodeTiled>(ptr);
  }
  return fn;
}

// 3-D bf16 tensor [T][H][inner] (inner contiguous), box [Q][1][inner], unswizzled.
// L2 fills no wider than one (token, head) row: a wider promotion pulls in
// the neighbouring head's row, which a balanced schedule reaches much later
// (after the line has left L2), so it would be read from HBM twice.
inline CUtensorMapL2promotion row_promotion(uint64_t row_bytes) {
  return row_bytes >= 256 ? CU_TENSOR_MAP_L2_PROMOTION_L2_256B
                          : (row_bytes >= 128 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_64B);
}

inline bool make_map_3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t H, uint64_t T, uint32_t Q) {
  PFN_encodeTiled enc = get_encode_tiled();
  if (!enc) return false;
  cuuint64_t dims[3] = {inner, H, T};
  cuuint64_t strides[2] = {inner * 2, inner * H * 2};
  cuuint32_t box[3] = {(cuuint32_t)inner, 1, Q};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, row_promotion(inner * 2),
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D bf16 tensor [T][H][R][inner] (inner contiguous), box [Q][1][R][64] with
// the 128-byte swizzle: each box lands as MR = Q*R rows of 128 B, exactly
// one 64-column block of a 128B-swizzled operand tile.
inline bool make_map_4d_sw128(CUtensorMap* m, const void* base, uint64_t inner, uint64_t R, uint64_t H,
                              uint64_t T, uint32_t Q) {
  PFN_encodeTiled enc = get_encode_tiled();
  if (!enc) return false;
  cuuint64_t dims[4] = {inner, R, H, T};
  cuuint64_t strides[3] = {inner * 2, inner * R * 2, inner * R * H * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)R, 1, Q};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, row_promotion(inner * R * 2),
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Stream-ordered memory for the balanced schedule's handover slots: a pool
// per device owned by the library that keeps what it has allocated (a few
// MB), so a call does not map fresh memory after every synchronisation.
inline cudaMemPool_t handover_pool(int dev) {
  static cudaMemPool_t pools[64] = {};
  static bool tried[64] = {};
  if (dev < 0 || dev >= 64) return nullptr;
  if (!tried[dev]) {
    tried[dev] = true;
    cudaMemPoolProps props{};
    props.allocType = cudaMemAllocationTypePinned;
    props.location.type = cudaMemLocationTypeDevice;
    props.location.id = dev;
    cudaMemPool_t pool = nullptr;
    if (cudaMemPoolCreate(&pool, &props) == cudaSuccess) {
      uint64_t keep = ~0ull;
      cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
      pools[dev] = pool;
    } else {
      cudaGetLastError();
    }
  }
  return pools[dev];
}

// Split schedule, between the two passes: the initial state of every piece
// of a unit, h_in(first) = the caller's state (zero without one) and
// h_in(next) = alpha * h_in(piece) + h_loc(piece), per pair and column,
// into the piece's handover slot.  Exact: the recurrence is affine in the
// state, and h_loc already holds the piece's carry term.  Block 0 of a
// unit also copies the caller's carry into the slot of the unit's first
// piece (the full pass overwrites the caller's with the unit's last token).
template <int N, int R, int Q>
__global__ void __launch_bounds__(256) split_combine_kernel(const ChunkParams p) {
  constexpr int K2 = N / 2, P = 64, KP = K2 * P;
  constexpr int kMaxPieces = 256;  // pieces of one unit (the launcher keeps ranges at most 148)
  __shared__ int sSlot[kMaxPieces];
  __shared__ int sCount;
  const int u = blockIdx.y;  // the unit; blockIdx.x: 256 of its K2 * P elements
  const int64_t nch = (p.L + Q - 1) / Q, total = (int64_t)p.bal_units * nch;
  if (threadIdx.x == 0) {  // the unit's pieces in order: the range holding its first chunk, then the next ones
    int k = (int)(u * nch * p.split_grid / total);
    while (k + 1 < p.split_grid && (int64_t)(k + 1) * total / p.split_grid <= u * nch) ++k;
    while (k > 0 && (int64_t)k * total / p.split_grid > u * nch) --k;
    int n = 0;
    for (; k < p.split_grid && n < kMaxPieces; ++k) {
      int3 pc[2];
      const int np = split_pieces(nch, total, p.split_grid, k, pc);
      int j = 0;
      while (j < np && pc[j].x != u) ++j;
      if (j == np) break;
      sSlot[n++] = 2 * k + j;
      if (pc[j].z == nch) break;  // the unit's last piece
    }
    sCount = n;
  }
  __syncthreads();
  if (blockIdx.x == 0 && sCount > 0) {  // the caller's carry, for the full pass of the unit's first piece
    const int64_t s0 = sSlot[0];
    if (p.prev_B)
      for (int i = threadIdx.x; i < R * N; i += blockDim.x) p.xB[s0 * R * N + i] = p.prev_B[(int64_t)u * R * N + i];
    if (p.prev_x)
      for (int i = threadIdx.x; i < R * P; i += blockDim.x) p.xx[s0 * R * P + i] = p.prev_x[(int64_t)u * R * P + i];
  }
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= KP) return;
  const int k2 = e / P;
  float2 h = p.h ? reinterpret_cast<const float2*>(p.h)[(int64_t)u * KP + e] : make_float2(0.f, 0.f);
  const int n = sCount;
  const float2* __restrict__ alpha = p.seg_alpha;
  const float2* __restrict__ hloc = reinterpret_cast<const float2*>(p.seg_h);
  float2* __restrict__ hin = reinterpret_cast<float2*>(p.xh);
  // four pieces' alpha and h_loc loaded ahead of their steps (the chain
  // through h is short arithmetic; the loads are not on it)
  for (int i0 = 0; i0 < n; i0 += 4) {
    float2 a[4], z[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = i0 + j;
      if (i + 1 < n) {
        a[j] = alpha[(int64_t)sSlot[i] * K2 + k2];
        z[j] = hloc[(int64_t)sSlot[i] * KP + e];
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int i = i0 + j;
      if (i < n) hin[(int64_t)sSlot[i] * KP + e] = h;
      if (i + 1 < n)
        h = make_float2(fmaf(a[j].x, h.x, fmaf(-a[j].y, h.y, z[j].x)), fmaf(a[j].x, h.y, fmaf(a[j].y, h.x, z[j].y)));
    }
  }
}

// Packed sequences, one CTA per unit: the sequences by length, longest
// first (ties by index), so that the block scheduler starts the longest
// units first and the short ones fill in behind them (longest processing
// time first).  One block; nseq <= kMaxOrderSeq.
constexpr int kMaxOrderSeq = 2048;
__global__ void __launch_bounds__(1024) seq_order_kernel(const int32_t* cu, int nseq, int32_t* order) {
  __shared__ int len[kMaxOrderSeq];
  for (int i = threadIdx.x; i < nseq; i += blockDim.x) len[i] = cu[i + 1] - cu[i];
  __syncthreads();
  for (int i = threadIdx.x; i < nseq; i += blockDim.x) {
    const int li = len[i];
    int rank = 0;
    for (int j = 0; j < nseq; ++j) rank += (len[j] > li) | ((len[j] == li) & (j < i));
    order[rank] = i;
  }
}

// fixed: caller-provided scratch (fixed_bytes long) for the handover slots
// instead of the pool; a request that needs more is refused.
template <int N, int R, int Q, bool RE>
m3_status chunked_launch(const m3_prefill_args* a, float* h, void* prev_B, void* prev_x, int nseq, cudaStream_t s,
                         void* fixed, size_t fixed_bytes) {
  using Cfg = ChunkCfg<N, R, Q, RE>;
  const int H = a->dims.nheads;
  const uint64_t T = (uint64_t)a->seqlen * (a->cu_seqlens ? 1 : a->dims.batch);
  CUtensorMap mx, mB, mC, mth;
  const int G = a->ngroups > 0 ? a->ngroups : H;
  if (!make_map_4d_sw128(&mx, a->x, 64, R, H, T, Q) || !make_map_4d_sw128(&mB, a->B, N, R, G, T, Q) ||
      !make_map_4d_sw128(&mC, a->C, N, R, G, T, Q))
    return M3_ERR_CUDA;
  if (RE) {
    mth = mx;  // not read: theta = 0
  } else if (!make_map_3d(&mth, a->theta, N / 2, H, T, Q)) {
    return M3_ERR_CUDA;
  }
  ChunkParams p{};
  p.x = static_cast<const __nv_bfloat16*>(a->x);
  p.B = static_cast<const __nv_bfloat16*>(a->B);
  p.dt = static_cast<const __nv_bfloat16*>(a->dt);
  p.lam = static_cast<const __nv_bfloat16*>(a->lam);
  p.A = a->A;
  p.D = a->D;
  p.cu_seqlens = a->cu_seqlens;
  p.y = a->y;
  p.ybf = a->y_dtype == M3_BF16;
  p.h = h;
  p.prev_B = static_cast<__nv_bfloat16*>(prev_B);
  p.prev_x = static_cast<__nv_bfloat16*>(prev_x);
  p.L = a->seqlen;
  p.H = H;
  p.G = G;
  p.pro = a->prologue;
  p.dt_bias = a->dt_bias;
  p.wait_ns = test_hooks().wait_ns.load();
  p.fault = test_hooks().fault.load();
  // X converted by the prologue warps at rank 1 without the BC norm (there
  // they have room for it; with the norm, at rank > 1 and in the split
  // schedule the state warps do it: measured faster each way)
  auto kern_sx = chunked_prefill_kernel<N, R, Q, RE>;
  auto kern = (R == 1 && !(a->prologue & M3_PRO_BC_NORM)) ? chunked_prefill_kernel<N, R, Q, RE, false, R == 1>
                                                          : kern_sx;
  if (cudaFuncSetAttribute(kern_sx, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) != cudaSuccess ||
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) != cudaSuccess)
    return M3_ERR_CUDA;
  const int units = nseq * H;
  // Split schedule: with fewer units than SMs (one long sequence of a few
  // heads), one CTA per unit leaves most SMs idle.  The units' chunks are
  // cut into one equal range per SM instead (a range holds the end of one
  // unit and the start of the next at most).  A state-only pass gives every
  // piece's own final state and total decay/rotation (all pieces in
  // parallel, no y), a small kernel chains them into each piece's exact
  // initial state (and copies the caller's carry for each unit's first
  // piece), and the full pass runs every piece from it.  At least
  // four chunks per range; not for packed batches or the no-allocation
  // entry point.
  {
    int dv = 0, nsm_s = 0;
    const int64_t nch = (a->seqlen + Q - 1) / Q;
    if (!fixed && !a->cu_seqlens && a->seqlen > 0 && cudaGetDevice(&dv) == cudaSuccess &&
        cudaDeviceGetAttribute(&nsm_s, cudaDevAttrMultiProcessorCount, dv) == cudaSuccess && units < nsm_s) {
      const int64_t total = (int64_t)units * nch;
      int grid = (int)(total / 4 < nsm_s ? total / 4 : nsm_s);
      if (grid > 256) grid = 256;  // (the combine's per-unit piece list)
      if (grid > units) {  // (so that no range is longer than a unit)
        const size_t nslot = 2 * (size_t)grid;
        const size_t hb = nslot * (size_t)(N / 2) * 64 * 2 * 4;
        size_t off = 0;
        auto take = [&](size_t bytes) {
          const size_t o = off;
          off += (bytes + 255) / 256 * 256;
          return o;
        };
        const size_t o_xh = take(hb), o_sh = take(hb), o_sa = take(nslot * (N / 2) * 8),
                     o_xB = take(nslot * R * N * 2), o_xx = take(nslot * R * 64 * 2);
        const size_t bytes = off;
        cudaMemPool_t pool = handover_pool(dv);
        void* buf = nullptr;
        auto kso = chunked_prefill_kernel<N, R, Q, RE, true>;
        if (pool && cudaFuncSetAttribute(kso, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) == cudaSuccess &&
            cudaMallocFromPoolAsync(&buf, bytes, pool, s) == cudaSuccess) {
          uint8_t* b8 = static_cast<uint8_t*>(buf);
          p.split_grid = grid;
          p.bal_units = units;
          p.xh = reinterpret_cast<float*>(b8 + o_xh);
          p.xB = reinterpret_cast<__nv_bfloat16*>(b8 + o_xB);
          p.xx = reinterpret_cast<__nv_bfloat16*>(b8 + o_xx);
          p.seg_h = reinterpret_cast<float*>(b8 + o_sh);
          p.seg_alpha = reinterpret_cast<float2*>(b8 + o_sa);
          kso<<<(unsigned)grid, Cfg::NT, Cfg::SMEM, s>>>(mx, mB, mC, mth, p);
          split_combine_kernel<N, R, Q><<<dim3((N / 2) * 64 / 256, (unsigned)units), 256, 0, s>>>(p);
          kern_sx<<<(unsigned)grid, Cfg::NT, Cfg::SMEM, s>>>(mx, mB, mC, mth, p);
          const cudaError_t e = cudaGetLastError();
          const cudaError_t ef = cudaFreeAsync(buf, s);
          record_launch(M3_TEST_KERNEL_CHUNKED_SPLIT, grid, (long long)bytes);
          return (e == cudaSuccess && ef == cudaSuccess) ? M3_OK : M3_ERR_CUDA;
        }
        cudaGetLastError();  // no pool memory: the one-CTA-per-unit launch below
      }
    }
  }
  // Balanced schedule: with more units than SMs, one CTA per unit leaves the
  // last wave partly empty (256 units on 148 SMs: the second wave is 73 %
  // full).  Instead every SM gets an equal range of the chunks, cutting at
  // most one unit at each end; fixed-length sequences only, a few whole
  // units per CTA at most.
  int dev = 0, nsm = 0, coop = 0, per_sm = 0;
  if (!a->cu_seqlens && a->seqlen > 0 && cudaGetDevice(&dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
      cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) == cudaSuccess && coop &&
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, Cfg::NT, Cfg::SMEM) == cudaSuccess &&
      per_sm >= 1) {
    const int grid = nsm * per_sm;
    const int64_t nch = (a->seqlen + Q - 1) / Q, total = (int64_t)units * nch;
    const int64_t range = (total + grid - 1) / grid;
    if (units > grid && total / grid >= nch && range <= (int64_t)(kMaxSeg - 2) * nch) {
      const size_t nslot = (size_t)grid + 1;
      const size_t off_xh = align_up((int)(nslot * 4), 256);
      const size_t off_xB = off_xh + nslot * (size_t)(N / 2) * 64 * 2 * 4;
      const size_t off_xx = off_xB + (size_t)align_up((int)(nslot * R * N * 2), 256);
      const size_t bytes = off_xx + nslot * (size_t)R * 64 * 2;
      void* buf = nullptr;
      if (fixed && bytes > fixed_bytes) return M3_ERR_SCRATCH;
      cudaMemPool_t pool = fixed ? nullptr : handover_pool(dev);
      if (fixed) buf = fixed;
      if (fixed || (pool && cudaMallocFromPoolAsync(&buf, bytes, pool, s) == cudaSuccess)) {
        uint8_t* b8 = static_cast<uint8_t*>(buf);
        p.bal_grid = grid;
        p.bal_units = units;
        p.xflag = reinterpret_cast<int*>(b8);
        p.xh = reinterpret_cast<float*>(b8 + off_xh);
        p.xB = reinterpret_cast<__nv_bfloat16*>(b8 + off_xB);
        p.xx = reinterpret_cast<__nv_bfloat16*>(b8 + off_xx);
        cudaError_t e = cudaMemsetAsync(p.xflag, 0, nslot * 4, s);
        if (e == cudaSuccess) {
          void* args[] = {&mx, &mB, &mC, &mth, &p};
          e = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(kern), dim3(grid), dim3(Cfg::NT), args,
                                          Cfg::SMEM, s);
        }
        const cudaError_t ef = fixed ? cudaSuccess : cudaFreeAsync(buf, s);
        record_launch(M3_TEST_KERNEL_CHUNKED_BALANCED, grid, (long long)bytes);
        return (e == cudaSuccess && ef == cudaSuccess) ? M3_OK : M3_ERR_CUDA;
      }
      cudaGetLastError();  // no pool memory: the one-CTA-per-unit launch below
    }
  }
  // packed sequences of different lengths on more units than SMs: the
  // longest units first (the order comes from the pool; without pool
  // memory, or with the caller's fixed scratch, the natural order)
  if (a->cu_seqlens && !fixed && nseq >= 2 && nseq <= kMaxOrderSeq) {
    int dv = 0, nsm_o = 0;
    void* buf = nullptr;
    cudaMemPool_t pool = nullptr;
    if (cudaGetDevice(&dv) == cudaSuccess &&
        cudaDeviceGetAttribute(&nsm_o, cudaDevAttrMultiProcessorCount, dv) == cudaSuccess && units > nsm_o &&
        (pool = handover_pool(dv)) != nullptr &&
        cudaMallocFromPoolAsync(&buf, (size_t)nseq * sizeof(int32_t), pool, s) == cudaSuccess) {
      p.seq_order = static_cast<const int32_t*>(buf);
      seq_order_kernel<<<1, 1024, 0, s>>>(a->cu_seqlens, nseq, static_cast<int32_t*>(buf));
      kern<<<units, Cfg::NT, Cfg::SMEM, s>>>(mx, mB, mC, mth, p);
      const cudaError_t e = cudaGetLastError();
      const cudaError_t ef = cudaFreeAsync(buf, s);
      record_launch(M3_TEST_KERNEL_CHUNKED, units, (long long)((size_t)nseq * sizeof(int32_t)));
      return (e == cudaSuccess && ef == cudaSuccess) ? M3_OK : M3_ERR_CUDA;
    }
    cudaGetLastError();
  }
  kern<<<units, Cfg::NT, Cfg::SMEM, s>>>(mx, mB, mC, mth, p);
  record_launch(M3_TEST_KERNEL_CHUNKED, units, 0);
  return cudaGetLastError() == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}

// Shapes with a chunked kernel: bf16 inputs, P = 64, and (N, R, chunk) in
// {(128, 1, 64), (64, 1, 64), (64, 4, 16), (64, 2, 32), (128, 2, 32)}; with
// theta = 0 (NULL) in {(128, 1, 64), (64, 1, 64), (64, 4, 16)}, without the
// BC norm.
inline m3_status chunked_prefill(const m3_prefill_args* a, float* h, void* prev_B, void* prev_x, int nseq,
                                 cudaStream_t s, void* fixed = nullptr, size_t fixed_bytes = 0) {
  const m3_dims& d = a->dims;
  if (d.in_dtype != M3_BF16 || d.headdim != 64) return M3_ERR_UNSUPPORTED;
  const int R = d.rank, N = d.dstate;
  const int Q = a->chunk > 0 ? a->chunk : (R == 1 ? 64 : 64 / R);
  const bool re = a->theta == nullptr;
  // the real-state variant feeds B and C to the MMAs as single f16 values,
  // exact only for the bf16 inputs themselves, not for normalised rows
  if (re && (a->prologue & M3_PRO_BC_NORM)) return M3_ERR_UNSUPPORTED;
#define M3_CH(NN, RR, QQ) \
  if (!re && N == NN && R == RR && Q == QQ)                                                  \
    return chunked_launch<NN, RR, QQ, false>(a, h, prev_B, prev_x, nseq, s, fixed, fixed_bytes);
#define M3_CH_RE(NN, RR, QQ) \
  if (re && N == NN && R == RR && Q == QQ)                                                   \
    return chunked_launch<NN, RR, QQ, true>(a, h, prev_B, prev_x, nseq, s, fixed, fixed_bytes);
  M3_CH_RE(128, 1, 64)
  M3_CH_RE(64, 1, 64)
  M3_CH_RE(64, 4, 16)
  M3_CH(128, 1, 64)
  M3_CH(64, 1, 64)
  M3_CH(64, 4, 16)
  M3_CH(64, 2, 32)
  M3_CH(128, 2, 32)
#undef M3_CH
#undef M3_CH_RE
  return M3_ERR_UNSUPPORTED;
}

}  // namespace m3
