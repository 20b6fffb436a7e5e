// gemm.cu -- grouped W4 GEMMs of the MoE layer on sm_103a tensor cores.
//
// The expert GEMMs take about 90% of prefill time (page "Revolutionizing Local
// AI Inference on Apple Silicon", section "Enhanced Tile and Scan
// Operations").  Weights stay 4-bit in HBM; each CTA streams one 128-row slice
// of packed codes with TMA, rebuilds it as fp16 one K-step at a time in tensor
// memory (w = scale*q + bias), and feeds tcgen05 MMAs that accumulate in FP32
// in tensor memory, so the expanded weights never reach HBM (page "Lily Beats
// MLX-LM 1.35x on Decode: Perplexity's Rust+Metal Engine for Apple Silicon",
// section "Prefill: fusing dequantisation and keeping routing GPU-resident").
//
// Operand roles (weights as the M=128 operand, token rows as N):
//   A = dequantised weight slice, 128 rows x 64 K per group, fp16, in tensor
//       memory (lane = weight row, two K elements per 32-bit column), written
//       by the dequant warps with tcgen05.st.  Gate/up: an item covers 64
//       features of both matrices; the 32 rows of TMEM lane quadrant q are
//       the gate rows of features 16q..16q+15, then the up rows of the same
//       features, so one MMA computes both projections of a feature, an item
//       needs one accumulator of N columns (two items' accumulators and a
//       deep A ring fit in tensor memory), and each epilogue warp finds the
//       gate and up outputs of its features in its own quadrant.  Down: 128
//       output features.
//   B = token rows of one block-map tile (<= BM rows) x 64 K, fp16, K-major,
//       128-byte swizzle, brought by TMA in boxes of up to 64 rows (one
//       128-row box when a BM 128 tile holds more than 64 rows): gate/up
//       reads xs, the fp16 rows of x in expert-sorted order written once per
//       layer by token_rows_kernel (one pass instead of a TMA gather per
//       K-step); down reads rows of H
//   D = 128 x N fp32 in TMEM
// Operand precision: fp16 rather than the pages' bf16.  Rounding the
// rebuilt weights and H to bf16 alone puts the layer outside max|err| <= 2e-2
// of rms on these weight distributions; fp16 is 8x finer, runs at the same
// kind::f16 tensor rate, and holds x, the group scales and biases exactly in
// [2^-17, 65504] (values beyond 65504 set LILY_STATUS_F16_RANGE).
// Epilogues: gate/up writes H = silu(g) * u (fp16) in expert-sorted row
// order; down writes its output rows as fp16 rows O (same order), staged
// through shared memory so that each lane stores 64 contiguous bytes of one
// row, and combine_kernel then sums each token's k + 1 rows, weighted by the
// routing gates, in a fixed order (the same bits on every run).
// K order: the rebuilt weights come out of the nibble extraction with each
// 8-element K chunk in the order (0,4,1,5,2,6,3,7); the K operands x16 and H
// are stored in that same order, so no shuffle is needed.
//
// Persistent: one CTA per SM walks the (tile, slice) work items; warp roles
// are listed below.  Every wait is bounded (2 s) and sets
// LILY_STATUS_TIMEOUT when it runs out.
#include "routing.cuh"

namespace lily {

// Warp roles.  Warp 0: TMA producer.  Warp 1: TMEM owner + MMA issuer (one
// thread).  Warps 2..9: dequant (one 128-row weight slice per K-step), which
// write the rebuilt weights straight into tensor memory (tcgen05.st): each
// warp owns the TMEM lane quadrant warp % 4, i.e. weight rows 32*(warp%4)..+31;
// warps 2..5 rebuild both quantisation groups of the even K-steps (of the
// CTA's running step count), 6..9 those of the odd ones, so two steps are
// rebuilt at once and each step is published by one set of four warps.  Warps 10..13: epilogue (TMEM -> global), overlapped with the next
// item's main loop through double-buffered accumulators; the epilogue warps
// also fill the next item's scale/bias table ahead of the dequant warps
// (gate/up; the down dequant lanes fill their own rows).
constexpr int kNumDequantWarps = 8;
constexpr int kNumEpiWarps = 4;
constexpr int kEpiWarp0 = 2 + kNumDequantWarps;
constexpr int kGemmThreads = 32 * (2 + kNumDequantWarps + kNumEpiWarps);  // 448
constexpr int kMaxStages = 12;
constexpr int kPackedBytes = 128 * 32;  // 128 rows x 64 4-bit codes
constexpr int kMaxA = 8;                // dequantised-A ring depth in K-steps (TMEM)
constexpr int kNumBars = 2 * kMaxStages + 2 * kMaxA + 4 + 4 + 1;

// Quantisation groups (64 K each) per K-step, two in both GEMMs: the fixed
// per-step hand-offs of every warp role (the producer's expect-tx and copies,
// the MMA warp's wait and commits, the dequant warps' waits, tensor-memory
// store wait and arrival) are paid once per 128 K.
__host__ __device__ constexpr int groups_per_step(bool /*gateup*/) { return 2; }

// 128-row weight sub-slices per work item (see GemmLayout::kSub): two at BM
// <= 64 (gate/up always; down when its d output features split into items of
// 256), else one.  nout: output features of each matrix (gate/up F, down d).
__host__ __device__ constexpr int sub_slices(bool gateup, int BM, int nout) {
  return BM > 64 ? 1 : (gateup || nout % 256 == 0) ? 2 : 1;
}

// Tensor memory (512 columns x 128 lanes): two accumulator sets of N <= BM
// columns, then the ring of dequantised A tiles (128 rows x 128 fp16 = 64
// columns per K-step).  A stage holds, per group, a 128-byte-swizzled tile of
// the token rows (BM x 64 fp16), and the packed codes of the step's 128
// weight rows (128 rows x 64 B, 64-byte swizzle; gate/up: the 64 gate rows of
// the slice, then its 64 up rows).
template <bool GATEUP, int BM, int SUB>
struct GemmLayout {
  static constexpr int kGroups = groups_per_step(GATEUP);
  static constexpr int kBTile = BM * 128;  // token rows of one group
  // token rows per TMA box: fewer, taller boxes per step (the rows past an
  // item's last are other tiles' rows or zero fill, never stored)
  static constexpr int kBoxRows = BM < 64 ? BM : 64;
  static constexpr int kBBytes = kGroups * kBTile;
  // 128-row sub-slices per item: tiles of at most 64 rows take two (gate/up:
  // 128 features of both matrices; down: 256 output features; 16 MMAs per
  // K-step), so the per-step hand-offs are paid once per two sub-slices and a
  // down item's token rows serve twice the features; BM 128 takes one, which
  // leaves room for two accumulator sets and a 4-step A ring
  static constexpr int kSub = SUB;
  static constexpr int kStage = kBBytes + kSub * kGroups * kPackedBytes;
  static constexpr int kOutRows = (GATEUP ? 64 : 128) * kSub;  // output features per item
  static constexpr int kACols = 32 * kGroups * kSub;          // A tiles of one K-step
  static constexpr int kAccCols = BM * kSub;                  // one accumulator set
  static constexpr int kNumAcc = 2;
  static constexpr int kAOff = kNumAcc * kAccCols;
  static constexpr int kNumA =
      (512 - kAOff) / kACols < kMaxA ? (512 - kAOff) / kACols : kMaxA;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kNumA >= 2, "tensor memory too small for the A ring");
  static_assert(SUB == 1 || (SUB == 2 && BM <= 64), "sub-slices");
};

// Down epilogue staging: per epilogue warp 32 rows x 32 output features of
// fp16, rows padded to 40 halves (80 bytes) so that the per-row 16-byte reads
// of eight consecutive rows hit eight different bank groups.
constexpr int kEpiRowHalves = 40;
constexpr int kEpiStageBytes = kNumEpiWarps * 32 * kEpiRowHalves * 2;
// At BM 128 the rows are packed (32 halves), the layout of a 32 x 32 box of
// O, so a full chunk leaves by one tensor store (partial chunks by the lanes).
template <int BM>
__host__ __device__ constexpr int epi_row_halves() { return BM == 128 ? 32 : kEpiRowHalves; }

// Gate/up: weight row r of an item (= TMEM lane r) is row code_row(r) of the
// step's code tile (64 gate rows, then 64 up rows): matrix (r >> 4) & 1 and
// feature 16 * (r >> 5) + (r & 15) of the item's 64.
__host__ __device__ constexpr int gu_matrix(int r) { return (r >> 4) & 1; }
__host__ __device__ constexpr int gu_feature(int r) { return 16 * (r >> 5) + (r & 15); }
__host__ __device__ constexpr int gu_code_row(int r) { return 64 * gu_matrix(r) + gu_feature(r); }

__host__ __device__ inline size_t gemm_fixed_bytes(bool gateup, int BM, int K, int nsb, int sub) {
  const int G = K / 64;
  return 1024                                    // alignment slack
         + (size_t)nsb * G * 128 * sub * 4       // scale/bias tables
         + (gateup ? 0 : kEpiStageBytes)          // down: epilogue staging
         + kNumBars * 8                          // mbarriers
         + 16;                                   // abort flag, TMEM address
}

size_t gemm_stage_bytes(bool gateup, int BM, int sub) {
  const int kg = groups_per_step(gateup);
  return (size_t)kg * ((size_t)BM * 128 + (size_t)sub * kPackedBytes);
}

constexpr size_t kSmemLimit = 232448;  // 227 KB per block

// Pipeline depth and scale-table buffering that fit in shared memory.
// Gate/up: two scale tables (the next item's is filled while the current one
// is in use) when that still leaves >= 3 stages, else one table.  Down: two
// tables always, one per dequant warp set.
static int stages_for(bool gateup, int BM, int K, int nsb, int sub) {
  const size_t fixed = gemm_fixed_bytes(gateup, BM, K, nsb, sub);
  if (fixed >= kSmemLimit) return 0;
  int s = (int)((kSmemLimit - fixed) / gemm_stage_bytes(gateup, BM, sub));
  return s > kMaxStages ? kMaxStages : s;
}

void gemm_config(bool gateup, int BM, int K, int sub, int* stages, int* nsb) {
  const int s2 = stages_for(gateup, BM, K, 2, sub);
  if (s2 >= 3 || (!gateup && s2 >= 2)) {  // down: one table per dequant warp set
    *stages = s2;
    *nsb = 2;
    return;
  }
  const int s1 = stages_for(gateup, BM, K, 1, sub);
  *stages = (gateup && s1 >= 2) ? s1 : 0;
  *nsb = 1;
}

int gemm_stages(bool gateup, int BM, int K, int nout) {
  int s, n;
  gemm_config(gateup, BM, K, sub_slices(gateup, BM, nout), &s, &n);
  return s;
}

size_t gemm_smem_bytes(bool gateup, int BM, int K, int sub) {
  int s, n;
  gemm_config(gateup, BM, K, sub, &s, &n);
  return gemm_fixed_bytes(gateup, BM, K, n, sub) + (size_t)s * gemm_stage_bytes(gateup, BM, sub);
}

// Position in a ring of n slots: slot index and the parity of its use count
// (it % n and (it / n) & 1 for the it-th use), advanced without a division.
struct Ring {
  uint32_t idx = 0, ph = 0;
  __device__ __forceinline__ void next(uint32_t n) {
    if (++idx == n) {
      idx = 0;
      ph ^= 1u;
    }
  }
};

// One work item = one block-map tile (or shared-expert tile) x one slice of
// output features (gate/up: 64 features of both matrices; down: 128).  Items
// are numbered tile-major so the slices of one tile, and the tiles of one
// expert, run at the same time and share the expert's weights and token rows
// through L2.  Shared-expert tiles come first.
struct Item {
  int expert, row0, rows, slice;
  bool shared;
};

// Item w from its tile's table entry {expert, row0, rows, 0} (written by the
// token-row kernel); false when the tile holds no rows.
__device__ __forceinline__ int4 load_tile(const GemmArgs& a, int w, int nslices) {
  return __ldg(a.tiles + w / nslices);
}
__device__ __forceinline__ bool item_from(int4 t, int w, int nslices, int nsh, Item& it) {
  it.slice = w % nslices;
  it.shared = w / nslices < nsh;
  it.expert = t.x;
  it.row0 = t.y;
  it.rows = t.z;
  return t.z > 0;
}

// Advance w (stepping by gridDim.x) to the next valid item; false at the end.
__device__ __forceinline__ bool next_item(const GemmArgs& a, int& w, int n_items, int nslices,
                                          int nsh, Item& it) {
  for (; w < n_items; w += gridDim.x)
    if (item_from(load_tile(a, w, nslices), w, nslices, nsh, it)) return true;
  return false;
}

// One scale-table word: fp16(scale) | fp16(bias) << 16 from bf16 bit patterns.
__device__ __forceinline__ uint32_t sb_word(uint16_t sc, uint16_t bi) {
  return (uint32_t)bf16_to_f16_bits(sc) | ((uint32_t)bf16_to_f16_bits(bi) << 16);
}

// Scale/bias table of one gate/up item: sb[g][r] = (fp16 scale | fp16 bias <<
// 16) of weight row r (128 rows per sub-slice, see gu_code_row) and every
// group g; `ld` words per group.  Filled by the epilogue threads, thread r
// owning rows r (+ 128 per further sub-slice) (`row` = its matrix row,
// `sp`/`bp` = its matrix's scales and biases): 16-byte loads of 8 scales and
// the 8 matching biases (two such pairs in flight), one f16x2 conversion and
// one 4-byte store per group.
__device__ void scale_fill(const uint16_t* sp, const uint16_t* bp, size_t row, int G, int r,
                           int ld, uint32_t* sbw) {
  if ((G & 7) == 0) {
    const int nch = G / 8;
    for (int base = 0; base < nch; base += 2) {
      uint4 vs[2], vb[2];
#pragma unroll
      for (int j = 0; j < 2; ++j)
        if (base + j < nch) {
          vs[j] = __ldg(reinterpret_cast<const uint4*>(sp + row * G) + base + j);
          vb[j] = __ldg(reinterpret_cast<const uint4*>(bp + row * G) + base + j);
        }
#pragma unroll
      for (int j = 0; j < 2; ++j)
        if (base + j < nch) {
          const uint32_t ws[4] = {vs[j].x, vs[j].y, vs[j].z, vs[j].w};
          const uint32_t wb[4] = {vb[j].x, vb[j].y, vb[j].z, vb[j].w};
          uint32_t* dst = sbw + (size_t)((base + j) * 8) * ld + r;
#pragma unroll
          for (int u = 0; u < 4; ++u) {  // groups 2u (low halves) and 2u+1 (high halves)
            const __half2 lo = __floats2half2_rn(__uint_as_float(ws[u] << 16),
                                                 __uint_as_float(wb[u] << 16));
            const __half2 hi = __floats2half2_rn(__uint_as_float(ws[u] & 0xFFFF0000u),
                                                 __uint_as_float(wb[u] & 0xFFFF0000u));
            dst[(2 * u) * ld] = *reinterpret_cast<const uint32_t*>(&lo);
            dst[(2 * u + 1) * ld] = *reinterpret_cast<const uint32_t*>(&hi);
          }
        }
    }
  } else {
    for (int g = 0; g < G; ++g)
      sbw[(size_t)g * ld + r] = sb_word(__ldg(sp + row * G + g), __ldg(bp + row * G + g));
  }
}

// Persistent kernel: one CTA per SM loops over the work items.
template <bool GATEUP, int BM, int SUB>
__global__ void __launch_bounds__(kGemmThreads, 1)
    w4_gemm_kernel(const __grid_constant__ CUtensorMap tm_q0,
                   const __grid_constant__ CUtensorMap tm_q1,
                   const __grid_constant__ CUtensorMap tm_b,
                   const __grid_constant__ CUtensorMap tm_b2,
                   const __grid_constant__ CUtensorMap tm_bw,
                   const __grid_constant__ CUtensorMap tm_b2w, const GemmArgs a, const int nstages,
                   const int nsb) {
  using L = GemmLayout<GATEUP, BM, SUB>;
  constexpr int BBYTES = L::kBBytes;
  constexpr int STAGE = L::kStage;
  constexpr int NACC = L::kNumAcc;
  // A buffers in use: at most the stage count.  A dequant warp at step it
  // knows only that the MMAs of step it - NA have finished; its parity wait
  // on the stage of step it is sound only if the stage's previous use (step
  // it - nstages) has landed, i.e. if nstages >= NA.
  const int NA = L::kNumA < nstages ? L::kNumA : nstages;

  const int K = GATEUP ? a.d : a.F;     // reduction length
  const int NOUT = GATEUP ? a.F : a.d;  // output features of each matrix
  constexpr int KG = L::kGroups;
  const int G = K / 64;                 // quantisation groups
  const int NST = G / KG;               // K-steps per item
  const int nslices = NOUT / L::kOutRows;
  const int P = a.T * a.k;
  const int nsh = (a.T + BM - 1) / BM;
  const int cap = (P + BM - 1) / BM + min(a.E, P);
  const int ntiles = min(max(*a.n_tiles, 0), cap);
  const int n_items = (nsh + ntiles) * nslices;

  // ---- shared memory carve-up
  extern __shared__ uint8_t smem_raw[];
  // aligned up to 1024 bytes by pointer arithmetic on the shared array, so
  // the compiler keeps the accesses in the shared window (not generic)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* stage_base = smem;
  uint32_t* sb = (uint32_t*)(smem + (size_t)nstages * STAGE);  // [nsb][G][128*SUB] scale|bias<<16
  const int sb_words = G * 128 * SUB;                        // one table
  uint8_t* estage = (uint8_t*)(sb + nsb * sb_words);         // epilogue staging
  uint64_t* bars = (uint64_t*)(estage + (GATEUP ? 0 : kEpiStageBytes));
  uint64_t* full = bars;                      // [kMaxStages] TMA landed
  uint64_t* empty = full + kMaxStages;        // [kMaxStages] stage consumed by the MMAs
  uint64_t* afull = empty + kMaxStages;       // [kMaxA] dequantised A ready in TMEM
  uint64_t* aempty = afull + kMaxA;           // [kMaxA] A consumed by the MMAs
  uint64_t* accfull = aempty + kMaxA;         // [2] accumulator set final
  uint64_t* accempty = accfull + 2;           // [2] accumulator set drained by the epilogue
  uint64_t* sbfull = accempty + 2;            // [2] scale table filled (epilogue -> dequant)
  uint64_t* sbempty = sbfull + 2;             // [2] scale table no longer read (dequant -> epilogue)
  uint64_t* drain = sbempty + 2;              // every MMA of this CTA finished
  int* misc = (int*)(drain + 1);
  volatile int* abort = misc;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- set-up
  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < kMaxA; ++b) {
      // one warp set per K-step (SUB 1) or all eight warps (SUB 2)
      mbar_init(smem_u32(&afull[b]), SUB == 1 ? kNumDequantWarps / 2 : kNumDequantWarps);
      mbar_init(smem_u32(&aempty[b]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&accfull[b]), 1);
      mbar_init(smem_u32(&accempty[b]), kNumEpiWarps);
      mbar_init(smem_u32(&sbfull[b]), kNumEpiWarps);
      mbar_init(smem_u32(&sbempty[b]), kNumDequantWarps);
    }
    mbar_init(smem_u32(drain), 1);
    misc[0] = 0;
    fence_mbar_init();
    prefetch_tensormap(&tm_q0);
    prefetch_tensormap(&tm_q1);  // gate/up: up codes; down: the output rows
    prefetch_tensormap(&tm_b);
    if (GATEUP) prefetch_tensormap(&tm_b2);
    if (BM > 64) {
      prefetch_tensormap(&tm_bw);
      if (GATEUP) prefetch_tensormap(&tm_b2w);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&misc[1]), L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = (uint32_t)misc[1];
  pdl_wait();  // the set-up above overlaps the predecessor; its outputs are read below
  pdl_trigger();

  if (warp == 0) {
    // ================================================= TMA producer
    uint32_t it = 0;  // K-steps issued by this CTA, across items
    Ring rs;          // stage ring position of step it
    bool ok = true;
    // the next item's table entry is loaded one item ahead (in every role)
    int4 tnext = (int)blockIdx.x < n_items ? load_tile(a, blockIdx.x, nslices) : make_int4(0, 0, 0, 0);
    for (int w = blockIdx.x; ok && w < n_items; w += gridDim.x) {
      const int4 tcur = tnext;
      if (w + (int)gridDim.x < n_items) tnext = load_tile(a, w + gridDim.x, nslices);
      Item itm;
      if (!item_from(tcur, w, nslices, nsh, itm)) {
        if (lane == 0) set_status(a.status, LILY_STATUS_BAD_TILE);
        continue;
      }
      const int N = (itm.rows + 15) & ~15;
      const int wrow = itm.expert * NOUT + itm.slice * L::kOutRows;
      // token rows of the item: gate/up reads the expert-sorted copy xs (or,
      // for a shared-expert tile, x16 in token order); down reads H
      // a tile of more than 64 rows (BM 128) takes one 128-row box per group
      const bool wide = BM > 64 && N > 64;
      const CUtensorMap* tmb = (GATEUP && itm.shared) ? (wide ? &tm_b2w : &tm_b2)
                                                      : (wide ? &tm_bw : &tm_b);
      const int brow = (GATEUP && itm.shared) ? itm.row0 - P : itm.row0;
      const int box_rows = wide ? BM : L::kBoxRows;
      const int nbox = wide ? 1 : (N + L::kBoxRows - 1) / L::kBoxRows;
      const uint32_t tx_bytes = KG * (SUB * kPackedBytes + nbox * box_rows * 128);
      for (int kk = 0; kk < NST; ++kk, ++it, rs.next(nstages)) {
        const int s = rs.idx;
        if (it >= (uint32_t)nstages &&
            !warp_wait_all(smem_u32(&empty[s]), rs.ph ^ 1u, abort, a.status)) {
          ok = false;
          break;
        }
        // whole warp, warp-uniform operands; one elected lane issues the step
        const uint32_t fb = smem_u32(&full[s]);
        const uint32_t st = smem_u32(stage_base + (size_t)s * STAGE);
        if (elect_one()) {
          mbar_arrive_expect_tx(fb, tx_bytes);
          // the step's packed codes, 128 rows x (KG * 32) bytes: gate/up
          // takes the slice's 64 gate rows, then the same features' up rows
#pragma unroll
          for (int j = 0; j < SUB; ++j) {  // sub-slice j: its code tile of 128 rows
            const uint32_t ct = st + BBYTES + j * KG * kPackedBytes;
            tma_load_2d(ct, &tm_q0, kk * KG * 32, wrow + (GATEUP ? 64 : 128) * j, fb);
            if (GATEUP) tma_load_2d(ct + 64 * KG * 32, &tm_q1, kk * KG * 32, wrow + 64 * j, fb);
          }
#pragma unroll
          for (int g = 0; g < KG; ++g) {
            const int grp = kk * KG + g;
            for (int rb = 0; rb < nbox; ++rb)  // the tile's N rows
              tma_load_2d(st + g * L::kBTile + rb * box_rows * 128, tmb, grp * 64,
                          brow + rb * box_rows, fb);
          }
        }
        __syncwarp();
      }
    }
    if (*abort && lane == 0) {  // let copies still in flight land before exit
      int never = 0;
      for (uint32_t k2 = (it > (uint32_t)nstages ? it - nstages : 0); k2 < it; ++k2)
        mbar_wait(smem_u32(&full[k2 % nstages]), (k2 / nstages) & 1, &never, a.status);
    }
  } else if (warp == 1) {
    // ================================================= MMA issuer
    // The whole warp runs the loop with warp-uniform operands; one elected
    // lane issues a K-step's MMAs and commits in one branch (measured faster
    // than an election per instruction).  It waits on afull alone: the dequant
    // warps arrive there only after their own wait on the stage's TMA
    // barrier, so a full A buffer implies that the stage's token rows landed.
    uint32_t it = 0, titem = 0;
    Ring rs;  // stage ring position of step it
    Ring ra;  // A ring position of step it
    bool ok = true;
    int4 tnext = (int)blockIdx.x < n_items ? load_tile(a, blockIdx.x, nslices) : make_int4(0, 0, 0, 0);
    for (int w = blockIdx.x; ok && w < n_items; w += gridDim.x) {
      const int4 tcur = tnext;
      if (w + (int)gridDim.x < n_items) tnext = load_tile(a, w + gridDim.x, nslices);
      Item itm;
      if (!item_from(tcur, w, nslices, nsh, itm)) continue;
      const int N = (itm.rows + 15) & ~15;
      const uint32_t idesc = idesc_f16_f32(128, N);
      const int ab = titem % NACC;
      if (titem >= (uint32_t)NACC &&
          !warp_wait_all(smem_u32(&accempty[ab]), ((titem / NACC) + 1) & 1, abort, a.status))
        break;
      tc_fence_after();
      const uint32_t dacc = tmem + ab * L::kAccCols;
      for (int kk = 0; kk < NST; ++kk, ++it, rs.next(nstages), ra.next(NA)) {
        const int s = rs.idx, b = ra.idx;
        if (!warp_wait_all(smem_u32(&afull[b]), ra.ph, abort, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sbase = smem_u32(stage_base + (size_t)s * STAGE);
        const uint32_t at = tmem + L::kAOff + b * L::kACols;  // A tile in TMEM
        if (elect_one()) {
#pragma unroll
          for (int g = 0; g < KG; ++g) {
            const uint64_t bdesc = sdesc_sw128(sbase + g * L::kBTile);
#pragma unroll
            for (int j = 0; j < SUB; ++j)  // sub-slice j: its A tile and accumulator
#pragma unroll
              for (int k16 = 0; k16 < 4; ++k16)  // +32 B along K = +2 in the descriptor
                mma_f16_ts(dacc + j * BM, at + j * 32 * KG + g * 32 + k16 * 8, bdesc + 2 * k16,
                           idesc, (kk | g | k16) != 0);
          }
          mma_commit(smem_u32(&empty[s]));
          mma_commit(smem_u32(&aempty[b]));
        }
        __syncwarp();
      }
      if (!ok) break;
      mma_commit_warp(smem_u32(&accfull[ab]));
      ++titem;
    }
    mma_commit_warp(smem_u32(drain));  // arrives once every MMA above has finished
    __syncwarp();
  } else if (warp < kEpiWarp0) {
    // ================================================= dequant
    // One sub-slice (SUB 1): warps 2..5 rebuild the K-steps with an even
    // running index it, 6..9 those with an odd one (both groups each).  Two
    // sub-slices (SUB 2): warps 2..5 rebuild sub-slice 0 of every step, 6..9
    // sub-slice 1.  One weight row per lane.
    const int q = warp & 3;
    const int r = q * 32 + lane;          // weight row within the slice = TMEM lane
    const uint32_t par = (uint32_t)(warp - 2) >> 2;  // step parity (SUB 1) / sub-slice (SUB 2)
    const int jsub = SUB == 2 ? (int)par : 0;
    const int crow = GATEUP ? gu_code_row(r) : r;  // its row of the step's code tile
    const uint32_t tlane = (uint32_t)(q * 32) << 16;
    uint32_t it = 0, j = 0;
    Ring rs;  // stage ring position of step it
    Ring ra;  // A ring position of step it
    bool ok = true;
    // down: each lane fills its own row's table entries (the groups of its
    // own K-steps) in its warp set's table slot (par), which only it reads;
    // the raw bf16 scales and biases of the next item are loaded one item
    // ahead, as 16-byte chunks, when G is 8 or 16 (else read one by one at
    // the item's start)
    constexpr int kPfChunks = 2;  // 8-group chunks held in registers
    uint4 pfs[kPfChunks], pfb[kPfChunks];
    int pf_w = -1;                // work item whose scales pfs/pfb hold
    auto sb_row = [&](int expert, int slice) {
      return (size_t)expert * NOUT + (size_t)slice * L::kOutRows + jsub * 128 + r;
    };
    auto down_prefetch = [&](int wn, int4 t) {
      // 16-byte chunks of 8 groups: whole chunks only (G a multiple of 8)
      if (GATEUP || (G & 7) != 0 || G > 8 * kPfChunks || t.z <= 0) return;
      const size_t row = sb_row(t.x, wn % nslices);
#pragma unroll
      for (int c = 0; c < kPfChunks; ++c)
        if (c * 8 < G) {
          pfs[c] = __ldg(reinterpret_cast<const uint4*>(a.s0 + row * G) + c);
          pfb[c] = __ldg(reinterpret_cast<const uint4*>(a.b0 + row * G) + c);
        }
      pf_w = wn;
    };
    // groups 2kk, 2kk+1 (K-step kk of an item starting at running step it0)
    // belong to this warp when (it0 + kk) has its parity
    auto down_fill = [&](int w, const Item& itm, uint32_t it0) {
      // this warp set's slot, entries [group][table row jsub * 128 + r]
      uint32_t* dst = sb + par * sb_words + jsub * 128;
      if (pf_w == w) {
#pragma unroll
        for (int c = 0; c < kPfChunks; ++c)
          if (c * 8 < G) {
            // groups c*8 + 2u and c*8 + 2u + 1 (K-step 4c + u) sit in the
            // two halves of word u of each chunk
            const uint32_t ws[4] = {pfs[c].x, pfs[c].y, pfs[c].z, pfs[c].w};
            const uint32_t wb[4] = {pfb[c].x, pfb[c].y, pfb[c].z, pfb[c].w};
#pragma unroll
            for (int u = 0; u < 4; ++u)
              if (SUB == 2 || ((it0 + (uint32_t)u) & 1u) == par) {
                dst[(c * 8 + 2 * u) * (128 * SUB) + r] = sb_word((uint16_t)ws[u], (uint16_t)wb[u]);
                dst[(c * 8 + 2 * u + 1) * (128 * SUB) + r] =
                    sb_word((uint16_t)(ws[u] >> 16), (uint16_t)(wb[u] >> 16));
              }
          }
      } else {
        const size_t row = sb_row(itm.expert, itm.slice);
        for (int grp = 0; grp < G; ++grp)
          if (SUB == 2 || ((it0 + (uint32_t)(grp >> 1)) & 1u) == par)
            dst[grp * (128 * SUB) + r] =
                sb_word(__ldg(a.s0 + row * G + grp), __ldg(a.b0 + row * G + grp));
      }
    };
    // table entries two items ahead: the next item's entry (for the scale
    // prefetch below) was requested one item earlier, not just now
    const int g1 = (int)gridDim.x;
    int4 tnext = (int)blockIdx.x < n_items ? load_tile(a, blockIdx.x, nslices) : make_int4(0, 0, 0, 0);
    int4 tnext2 = (int)blockIdx.x + g1 < n_items ? load_tile(a, blockIdx.x + g1, nslices)
                                                 : make_int4(0, 0, 0, 0);
    for (int w = blockIdx.x; ok && w < n_items; w += g1) {
      const int4 tcur = tnext;
      tnext = tnext2;  // item w + g1
      if (w + 2 * g1 < n_items) tnext2 = load_tile(a, w + 2 * g1, nslices);
      Item itm;
      if (!item_from(tcur, w, nslices, nsh, itm)) continue;
      const int slot = GATEUP ? j % nsb : (int)par;
      if (GATEUP) {
        if (!warp_wait(smem_u32(&sbfull[slot]), (j / nsb) & 1, abort, a.status)) break;
      } else {
        down_fill(w, itm, it);
        if (w + (int)gridDim.x < n_items) down_prefetch(w + gridDim.x, tnext);
      }
      const uint32_t* sbs = sb + slot * sb_words;
      for (int kk = 0; kk < NST; ++kk, ++it, rs.next(nstages), ra.next(NA)) {
        if (SUB == 1 && (it & 1u) != par) continue;  // the other warp set's step
        const int s0 = rs.idx, b0 = ra.idx;
        // the stage's TMA landed and the A buffer was consumed; the warp
        // sleeps in the wait (it issues nothing while the epilogue warps,
        // which share its SM sub-partition, drain the accumulators)
        if (!warp_wait_all2_blocking(smem_u32(&full[s0]), rs.ph, smem_u32(&aempty[b0]),
                                     ra.ph ^ 1u, it >= (uint32_t)NA, abort, a.status)) {
          ok = false;
          break;
        }
        // the stage holds the step's codes as rows of 64 bytes (two groups)
        // with the 64-byte TMA swizzle: 16-byte chunk c of row R sits at
        // 16 * (c ^ ((R >> 1) & 3)), which spreads each 8 consecutive lanes'
        // loads (8 consecutive code rows) over all eight 16-byte bank groups
        const int ph = (crow >> 1) & 3;
        const uint8_t* pk = stage_base + (size_t)s0 * STAGE + BBYTES +
                            jsub * KG * kPackedBytes + crow * (KG * 32);
        const uint4 lo0 = *reinterpret_cast<const uint4*>(pk + 16 * (0 ^ ph));
        const uint4 hi0 = *reinterpret_cast<const uint4*>(pk + 16 * (1 ^ ph));
        const uint4 lo1 = *reinterpret_cast<const uint4*>(pk + 16 * (2 ^ ph));
        const uint4 hi1 = *reinterpret_cast<const uint4*>(pk + 16 * (3 ^ ph));
        const int tr = jsub * 128 + r;  // table row
        const uint32_t sbv0 = sbs[(kk * KG) * (128 * SUB) + tr];
        const uint32_t sbv1 = sbs[(kk * KG + 1) * (128 * SUB) + tr];
        const uint32_t s20 = prmt(sbv0, sbv0, 0x1010u), b20 = prmt(sbv0, sbv0, 0x3232u);
        const uint32_t s21 = prmt(sbv1, sbv1, 0x1010u), b21 = prmt(sbv1, sbv1, 0x3232u);
        const uint32_t wd0[8] = {lo0.x, lo0.y, lo0.z, lo0.w, hi0.x, hi0.y, hi0.z, hi0.w};
        const uint32_t wd1[8] = {lo1.x, lo1.y, lo1.z, lo1.w, hi1.x, hi1.y, hi1.z, hi1.w};
        uint32_t o0[32], o1[32];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {  // the two groups' arithmetic interleaved
          uint32_t t4[4], u4[4];
          dequant8(wd0[jj], s20, b20, t4);
          dequant8(wd1[jj], s21, b21, u4);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            o0[4 * jj + e] = t4[e];
            o1[4 * jj + e] = u4[e];
          }
        }
        const uint32_t acol = tmem + tlane + L::kAOff + b0 * L::kACols + jsub * 32 * KG;
        tmem_st32(acol, o0);
        tmem_st32(acol + 32, o1);
        // the stores must be complete before the MMA issuer is told: wait,
        // order them before the arrive, then one arrive per warp and step
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&afull[b0]));
      }
      if (!ok) break;
      __syncwarp();
      if (GATEUP && lane == 0) mbar_arrive(smem_u32(&sbempty[slot]));
      ++j;
    }
  } else {
    // ================================================= epilogue
    // Per item j: (1) gate/up: fill the scale table of item j+1 for the
    // dequant warps, (2) drain item j's accumulators to global memory.
    const int q = warp & 3;  // TMEM lane quadrant of this warp
    const int r = threadIdx.x - 32 * kEpiWarp0;
    auto slot_ptr = [&](int slot) { return sb + (size_t)slot * sb_words; };
    // gate/up: thread r fills the table entries of weight row r
    auto fill = [&](const Item& it, int slot) {
#pragma unroll
      for (int j = 0; j < SUB; ++j) {  // sub-slice j: table rows 128 j + r
        const size_t row = (size_t)it.expert * NOUT + (size_t)it.slice * L::kOutRows + 64 * j +
                           gu_feature(r);
        if (gu_matrix(r) == 0)
          scale_fill(a.s0, a.b0, row, G, 128 * j + r, 128 * SUB, slot_ptr(slot));
        else
          scale_fill(a.s1, a.b1, row, G, 128 * j + r, 128 * SUB, slot_ptr(slot));
      }
    };
    int w = blockIdx.x;
    Item cur, nxt, nn;
    bool have = next_item(a, w, n_items, nslices, nsh, cur);
    if (GATEUP && have) {
      fill(cur, 0);
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sbfull[0]));
    }
    int wn = w + gridDim.x;
    bool have_next = have && next_item(a, wn, n_items, nslices, nsh, nxt);
    // table entry of the item after next, requested one item ahead so that
    // its load is not waited for at the item boundary
    int4 tpre = (have_next && wn + (int)gridDim.x < n_items)
                    ? load_tile(a, wn + gridDim.x, nslices)
                    : make_int4(0, 0, 0, 0);
    uint32_t j = 0;
    while (have) {
      if (GATEUP && have_next) {
        const uint32_t jn = j + 1;
        const int slot = jn % nsb;
        if (jn >= (uint32_t)nsb &&
            !warp_wait(smem_u32(&sbempty[slot]), ((jn / nsb) + 1) & 1, abort, a.status))
          break;
        fill(nxt, slot);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sbfull[slot]));
      }
      int wnn = wn + gridDim.x;
      bool have_nn = false;
      if (have_next && wnn < n_items) {
        have_nn = item_from(tpre, wnn, nslices, nsh, nn);
        if (!have_nn) {  // an empty tile: scan on (rare)
          wnn += gridDim.x;
          have_nn = next_item(a, wnn, n_items, nslices, nsh, nn);
        }
      }
      if (have_nn && wnn + (int)gridDim.x < n_items) tpre = load_tile(a, wnn + gridDim.x, nslices);

      const int N = (cur.rows + 15) & ~15;
      const int ab = j % NACC;
      if (!warp_wait(smem_u32(&accfull[ab]), (j / NACC) & 1, abort, a.status)) break;
      tc_fence_after();
      const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16) + ab * L::kAccCols;
      bool range_ok = true;
      // 32-row chunks of each sub-slice's accumulator (columns js * BM + cb)
      const int nch = (N + 31) / 32;
      for (int ci = 0; ci < SUB * nch; ++ci) {
        const int js = SUB == 1 ? 0 : ci / nch, cb = 32 * (SUB == 1 ? ci : ci % nch);
        const bool last = ci == SUB * nch - 1;
        const int ncol = N - cb < 32 ? N - cb : 32;  // 16 or 32
        if (GATEUP) {
          // Lanes 0..15 of warp q hold the gate outputs g of features
          // 16q..16q+15 of the slice, lanes 16..31 the up outputs u of the
          // same features (32 rows each).  Per step lanes 0..15 compute H of
          // rows cb + rr and lanes 16..31 of rows cb + 16 + rr, each fetching
          // the other half's value of its row with one shuffle.
          uint32_t v[32];
          tmem_ld32(tl + js * BM + cb, v);
          tmem_ld_wait();
          if (last) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&accempty[ab]));
          }
          const bool hi = lane >= 16;
          const int feat = cur.slice * L::kOutRows + 64 * js + gu_feature(q * 32 + lane);
          // H holds each 8-feature chunk in K-chunk order (it is the down
          // GEMM's K operand against weights rebuilt in that order), so
          // features e and e + 4 sit side by side: lanes with e < 4 store the
          // pair of row rr, lanes with e >= 4 that of row rr + 1, one 4-byte
          // store each
          const bool up4 = (lane & 4) != 0;
          __half2* Hp = reinterpret_cast<__half2*>(static_cast<__half*>(a.H) +
                                                   ((feat & ~7) | ((feat & 3) << 1)));
          const int rb0 = cb + (hi ? 16 : 0);
#pragma unroll
          for (int rr = 0; rr < 16; rr += 2) {
            float hv[2];
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const uint32_t send = hi ? v[rr + t] : v[rr + t + 16];
              const float other = __uint_as_float(__shfl_xor_sync(0xffffffffu, send, 16));
              const float own = __uint_as_float(hi ? v[rr + t + 16] : v[rr + t]);
              const float gv = hi ? other : own, uv = hi ? own : other;
              // silu(g) * u with the fast reciprocal: its few-ulp fp32 error
              // is far below the fp16 rounding of H; g -> -inf gives 0
              hv[t] = __fdividef(gv, 1.f + __expf(-gv)) * uv;
            }
            const float recv = __shfl_xor_sync(0xffffffffu, up4 ? hv[0] : hv[1], 4);
            const float lo = up4 ? recv : hv[0], hi2 = up4 ? hv[1] : recv;
            const int n = rb0 + rr + (up4 ? 1 : 0);
            if (n < cur.rows) {
              range_ok &= fabsf(lo) <= 65504.f && fabsf(hi2) <= 65504.f;
              Hp[(size_t)(cur.row0 + n) * (a.F / 2)] = __floats2half2_rn(lo, hi2);
            }
          }
        } else {
          // Output rows of the item as fp16 into O, in the same
          // expert-sorted row order as H; the combine kernel then sums each
          // token's rows.  Each warp stages its 32 features of up to 32 rows
          // in shared memory; at BM 128 a chunk of 32 rows leaves as one
          // tensor store (tm_q1 is then O's map), else each lane stores one
          // row's 64 bytes.
          constexpr int RH = epi_row_halves<BM>();
          const int feat = cur.slice * L::kOutRows + js * 128 + q * 32 + lane;
          uint32_t va[16], vb[16];
          tmem_ld16(tl + js * BM + cb, va);
          if (ncol == 32) tmem_ld16(tl + js * BM + cb + 16, vb);
          tmem_ld_wait();
          if (last) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&accempty[ab]));
          }
          __half* buf = reinterpret_cast<__half*>(estage) + (size_t)q * 32 * kEpiRowHalves;
          if (BM == 128) {  // the previous chunk's tensor store has read the buffer
            if (lane == 0) bulk_wait_read();
            __syncwarp();
          }
#pragma unroll
          for (int rr = 0; rr < 16; ++rr) {
            const float v = __uint_as_float(va[rr]);
            range_ok &= fabsf(v) <= 65504.f;
            buf[rr * RH + lane] = __float2half_rn(v);
          }
          if (ncol == 32) {
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
              const float v = __uint_as_float(vb[rr]);
              range_ok &= fabsf(v) <= 65504.f;
              buf[(16 + rr) * RH + lane] = __float2half_rn(v);
            }
          }
          if (BM == 128 && ncol == 32 && cb + 32 <= cur.rows) {
            fence_proxy_async_shared();  // the stores above, to the tensor store
            __syncwarp();
            if (lane == 0) tma_store_2d(&tm_q1, feat - lane, cur.row0 + cb, smem_u32(buf));
          } else {
            __syncwarp();
            if (lane < ncol && cb + lane < cur.rows) {
              const uint4* src = reinterpret_cast<const uint4*>(buf + lane * RH);
              uint4* dst = reinterpret_cast<uint4*>(static_cast<__half*>(a.O) +
                                                    (size_t)(cur.row0 + cb + lane) * a.d +
                                                    (feat - lane));
              const uint4 v0 = src[0], v1 = src[1], v2 = src[2], v3 = src[3];
              dst[0] = v0;
              dst[1] = v1;
              dst[2] = v2;
              dst[3] = v3;
            }
            __syncwarp();
          }
        }
      }
      if (!range_ok) set_status(a.status, LILY_STATUS_F16_RANGE);
      cur = nxt;
      have = have_next;
      nxt = nn;
      wn = wnn;
      have_next = have_nn;
      ++j;
    }
    if (!GATEUP && BM == 128 && lane == 0) bulk_wait_all();  // O fully written
  }

  // ---- teardown: every MMA has finished before TMEM is released
  if (warp == 1 && lane == 0) {
    int never = 0;
    mbar_wait(smem_u32(drain), 0, &never, a.status);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, L::kTmemCols);
  }
}

// =================================================================== host side

CUresult encode_tiled(CUtensorMap* tm, CUtensorMapDataType dt, uint32_t rank, void* base,
                      const uint64_t* dims, const uint64_t* strides, const uint32_t* box,
                      CUtensorMapSwizzle swz) {
  using Fn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                          const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                          CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                          CUtensorMapFloatOOBfill);
  static Fn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !p)
      return CUDA_ERROR_NOT_FOUND;
    fn = (Fn)p;
  }
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return fn(tm, dt, rank, base, (const cuuint64_t*)dims, (const cuuint64_t*)strides,
            (const cuuint32_t*)box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

template <bool GATEUP, int BM, int SUB>
static cudaError_t launch_gemm_bm(const GemmArgs& a, const CUtensorMap& q0, const CUtensorMap& q1,
                                  const CUtensorMap& b, const CUtensorMap& b2,
                                  const CUtensorMap& bw, const CUtensorMap& b2w, cudaStream_t s) {
  const int K = GATEUP ? a.d : a.F;
  const int NOUT = GATEUP ? a.F : a.d;
  int nstages = 0, nsb = 0;
  gemm_config(GATEUP, BM, K, SUB, &nstages, &nsb);
  if (nstages < 2) return cudaErrorInvalidValue;
  const size_t smem = gemm_smem_bytes(GATEUP, BM, K, SUB);
  auto kern = w4_gemm_kernel<GATEUP, BM, SUB>;
  cudaError_t err = ensure_smem_attr((const void*)kern, smem);
  if (err != cudaSuccess) return err;
  const int P = a.T * a.k;
  const int cap = (P + BM - 1) / BM + (a.E < P ? a.E : P);
  const int nsh = (a.T + BM - 1) / BM;
  const int max_items = (nsh + cap) * (NOUT / GemmLayout<GATEUP, BM, SUB>::kOutRows);
  int num_sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    num_sms = 148;
  const int grid = max_items < num_sms ? max_items : num_sms;  // persistent: one CTA per SM
  prof_begin(GATEUP ? K_GATEUP : K_DOWN, s);
  err = launch_pdl(kern, dim3(grid), dim3(kGemmThreads), smem, s, q0, q1, b, b2, bw, b2w, a, nstages,
                   nsb);
  prof_end(GATEUP ? K_GATEUP : K_DOWN, s);
  return err;
}

template <bool GATEUP>
static cudaError_t launch_gemm(const GemmArgs& a, const CUtensorMap& q0, const CUtensorMap& q1,
                               const CUtensorMap& b, const CUtensorMap& b2, const CUtensorMap& bw,
                               const CUtensorMap& b2w, cudaStream_t s) {
  // gate/up: two sub-slices at BM <= 64; down: two when d splits into
  // 256-feature items, else one
  const bool two = sub_slices(GATEUP, a.BM, GATEUP ? a.F : a.d) == 2;
  switch (a.BM) {
#define LILY_GEMM_BM(BMV)                                                   \
  case BMV:                                                                 \
    if constexpr (GATEUP) {                                                 \
      return launch_gemm_bm<GATEUP, BMV, 2>(a, q0, q1, b, b2, bw, b2w, s);  \
    } else {                                                                \
      return two ? launch_gemm_bm<GATEUP, BMV, 2>(a, q0, q1, b, b2, bw, b2w, s) \
                 : launch_gemm_bm<GATEUP, BMV, 1>(a, q0, q1, b, b2, bw, b2w, s); \
    }
    LILY_GEMM_BM(16)
    LILY_GEMM_BM(32)
    LILY_GEMM_BM(64)
#undef LILY_GEMM_BM
    case 128: return launch_gemm_bm<GATEUP, 128, 1>(a, q0, q1, b, b2, bw, b2w, s);
    default: return cudaErrorInvalidValue;
  }
}

// Packed codes: boxes of box_rows rows x 64 bytes (the two quantisation
// groups of a K-step) with the 64-byte swizzle (the four 16-byte chunks of
// row r are permuted by XOR with (r >> 1) & 3), so that the dequant lanes'
// 16-byte loads are free of bank conflicts: per K-step one 128-row copy
// (down), or 64 rows of the gate matrix and 64 of the up matrix (gate/up).
static_assert(groups_per_step(true) == 2 && groups_per_step(false) == 2, "64-byte code rows");
static bool packed_map(CUtensorMap* tm, const uint8_t* q, int K, int rows, int box_rows) {
  uint64_t dims[2] = {(uint64_t)K / 2, (uint64_t)rows};
  uint64_t strides[1] = {(uint64_t)K / 2};
  uint32_t box[2] = {64, (uint32_t)box_rows};
  return encode_tiled(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, (void*)q, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_64B) == CUDA_SUCCESS;
}

// Token rows per TMA box (GemmLayout::kBoxRows).
static int box_rows(int BM) { return BM < 64 ? BM : 64; }

static bool f16_rows_map(CUtensorMap* tm, const void* base, int cols, int rows, int box_rows) {
  uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows};
  uint64_t strides[1] = {(uint64_t)cols * 2};
  uint32_t box[2] = {64, (uint32_t)box_rows};
  return encode_tiled(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, (void*)base, dims, strides, box,
                      CU_TENSOR_MAP_SWIZZLE_128B) == CUDA_SUCCESS;
}

// Token rows of the gate/up GEMM, one warp per output row: rows [0, P) of
// xs are x[perm[r] / k] (expert-sorted), rows of x16 are x in token order;
// both fp16, each 8-element chunk in K-chunk order.  Values beyond the fp16
// range set LILY_STATUS_F16_RANGE.
__global__ void __launch_bounds__(256) token_rows_kernel(const uint4* __restrict__ x,
                                                         const int32_t* __restrict__ perm, int k,
                                                         int P, int T, int d8, uint4* __restrict__ xs,
                                                         uint4* __restrict__ x16, uint32_t* status,
                                                         const GemmArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();  // routing (perm, block map) comes from the predecessor
  pdl_trigger();
  // tile table: {expert, row0, rows, 0}, shared-expert tiles first
  const int nsh = (T + a.BM - 1) / a.BM;
  const int ntab = tile_count(T, a.E, k, a.BM);
  const int cap = ntab - nsh;
  const int ntiles = min(max(*a.n_tiles, 0), cap);
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < ntab; t += gridDim.x * blockDim.x) {
    int4 v = make_int4(0, 0, 0, 0);
    if (t < nsh) {
      v = make_int4(a.E, P + t * a.BM, min(a.BM, T - t * a.BM), 0);
    } else if (t - nsh < ntiles) {
      const int e = __ldg(a.block_map + 2 * (t - nsh)), row0 = __ldg(a.block_map + 2 * (t - nsh) + 1);
      if (e >= 0 && e < a.E && row0 >= 0 && row0 < P) {
        const int rows = min(min(a.BM, __ldg(a.offsets + e + 1) - row0), P - row0);
        if (rows > 0) v = make_int4(e, row0, rows, 0);
      } else {
        set_status(a.status, LILY_STATUS_BAD_TILE);
      }
    }
    a.tiles[t] = v;
  }
  bool ok = true;
  for (int row = blockIdx.x * 8 + warp; row < P + T; row += gridDim.x * 8) {
    int tok = row - P;
    if (row < P) {
      const int p = __ldg(perm + row);
      if (p < 0 || p >= P) {  // not a permutation entry: flagged, row 0 used
        if (lane == 0) set_status(status, LILY_STATUS_BAD_TILE);
      }
      tok = min(max(p, 0), P - 1) / k;
    }
    const uint4* src = x + (size_t)tok * d8;
    uint4* dst = row < P ? xs + (size_t)row * d8 : x16 + (size_t)(row - P) * d8;
    // up to eight loads of the row in flight per lane before the stores
    constexpr int kU = 8;
    for (int c0 = lane; c0 < d8; c0 += 32 * kU) {
      uint4 v[kU];
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (c0 + 32 * u < d8) v[u] = __ldg(src + c0 + 32 * u);
#pragma unroll
      for (int u = 0; u < kU; ++u)
        if (c0 + 32 * u < d8) dst[c0 + 32 * u] = bf8_to_h8_kchunk(v[u], ok);
    }
  }
  if (!ok) set_status(status, LILY_STATUS_F16_RANGE);
}

cudaError_t launch_token_rows(const GemmArgs& a, const void* x, void* xs, void* x16,
                              cudaStream_t s) {
  const int P = a.T * a.k;
  int blocks = (P + a.T + 7) / 8;
  const int tb = (tile_count(a.T, a.E, a.k, a.BM) + 255) / 256;
  if (blocks < tb) blocks = tb;
  if (blocks > 152 * 8) blocks = 152 * 8;
  prof_begin(K_TOKEN_ROWS, s);
  const cudaError_t err = launch_pdl(token_rows_kernel, dim3(blocks), dim3(256), 0, s,
                                     static_cast<const uint4*>(x), a.perm, a.k, P, a.T, a.d / 8,
                                     static_cast<uint4*>(xs), static_cast<uint4*>(x16), a.status, a);
  prof_end(K_TOKEN_ROWS, s);
  return err;
}

cudaError_t launch_gateup(const GemmArgs& a, const void* xs, const void* x16, const uint8_t* gq,
                          const uint8_t* uq, cudaStream_t s) {
  CUtensorMap q0, q1, b, b2, bw, b2w;
  const int P = a.T * a.k;
  if (!packed_map(&q0, gq, a.d, (a.E + 1) * a.F, 64) ||
      !packed_map(&q1, uq, a.d, (a.E + 1) * a.F, 64) ||
      !f16_rows_map(&b, xs, a.d, P, box_rows(a.BM)) ||
      !f16_rows_map(&b2, x16, a.d, a.T, box_rows(a.BM)) ||
      !f16_rows_map(&bw, xs, a.d, P, a.BM) || !f16_rows_map(&b2w, x16, a.d, a.T, a.BM))
    return cudaErrorInvalidValue;
  return launch_gemm<true>(a, q0, q1, b, b2, bw, b2w, s);
}

cudaError_t launch_down(const GemmArgs& a, const uint8_t* dq, cudaStream_t s) {
  CUtensorMap q0, b, bw, o;
  const int P = a.T * a.k;
  // o: the output rows O, 32 x 32 boxes without swizzle (the epilogue's
  // staging layout at BM 128), for the tensor stores of full chunks
  uint64_t odims[2] = {(uint64_t)a.d, (uint64_t)(P + a.T)};
  uint64_t ostrides[1] = {(uint64_t)a.d * 2};
  uint32_t obox[2] = {32, 32};
  if (!packed_map(&q0, dq, a.F, (a.E + 1) * a.d, 128) ||
      !f16_rows_map(&b, a.H, a.F, P + a.T, box_rows(a.BM)) ||
      !f16_rows_map(&bw, a.H, a.F, P + a.T, a.BM) ||
      encode_tiled(&o, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, a.O, odims, ostrides, obox,
                   CU_TENSOR_MAP_SWIZZLE_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  return launch_gemm<false>(a, q0, o, b, b, bw, bw, s);
}

// Combine: y[t] = sum_j gate[t][j] * O[inv[t*k + j]] + O[P + t] (the k
// routed rows of token t in slot order, weighted by their routing gates, then
// its shared-expert row), in fp32 and in that fixed order, so the layer
// output is the same on every run.  One CTA per
// token; each thread takes 8 consecutive outputs and issues the loads of all
// k + 1 rows before adding.  Modes: y fp32, y bf16, or the stacked prefill's
// boundary: x[t] += y[t] (fp32 residual) and, when xn is given, xn[t] =
// bf16(x[t] / sqrt(mean(x[t]^2) + eps)) for the next layer.
constexpr int kCombThreads = 256;
template <int MODE>  // 0: y fp32, 1: y bf16, 2: residual
__global__ void __launch_bounds__(kCombThreads) combine_kernel(
    const __half* __restrict__ O, const int32_t* __restrict__ inv,
    const float* __restrict__ gates, int k, int P, int d, void* y, float* x, __nv_bfloat16* xn,
    float eps, uint32_t* status) {
  __shared__ float s_red[kCombThreads / 32];
  pdl_wait();  // O comes from the down GEMM
  pdl_trigger();
  const int t = blockIdx.x;
  int rows[kMaxK + 1];
  float gw[kMaxK + 1];
  bool bad = false;
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    int r = 0;
    gw[j] = 0.f;
    if (j < k) {
      r = __ldg(inv + (size_t)t * k + j);
      gw[j] = __ldg(gates + (size_t)t * k + j);
      bad |= r < 0 || r >= P;
      r = min(max(r, 0), P - 1);
    }
    rows[j] = r;
  }
  gw[kMaxK] = 1.f;  // the shared expert
  if (bad && threadIdx.x == 0) set_status(status, LILY_STATUS_BAD_TILE);
  rows[kMaxK] = P + t;
  const int d8 = d / 8;
  float ss = 0.f;
  for (int c = threadIdx.x; c < d8; c += kCombThreads) {
    uint4 v[kMaxK + 1];
#pragma unroll
    for (int j = 0; j <= kMaxK; ++j)
      if (j < k || j == kMaxK)
        v[j] = __ldcs(reinterpret_cast<const uint4*>(O + (size_t)rows[j] * d) + c);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j <= kMaxK; ++j) {
      if (j < k || j == kMaxK) {
        const __half2* h = reinterpret_cast<const __half2*>(&v[j]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(h[e]);
          acc[2 * e] = fmaf(gw[j], f.x, acc[2 * e]);
          acc[2 * e + 1] = fmaf(gw[j], f.y, acc[2 * e + 1]);
        }
      }
    }
    const size_t o = (size_t)t * d + (size_t)c * 8;
    if (MODE == 0) {
      float4* yo = reinterpret_cast<float4*>(static_cast<float*>(y) + o);
      yo[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      yo[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else if (MODE == 1) {
      __nv_bfloat162 b[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) b[e] = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(y) + o) =
          *reinterpret_cast<const uint4*>(b);
    } else {
      float4* xo = reinterpret_cast<float4*>(x + o);
      float4 a0 = xo[0], a1 = xo[1];
      a0.x += acc[0]; a0.y += acc[1]; a0.z += acc[2]; a0.w += acc[3];
      a1.x += acc[4]; a1.y += acc[5]; a1.z += acc[6]; a1.w += acc[7];
      xo[0] = a0;
      xo[1] = a1;
      ss = fmaf(a0.x, a0.x, ss); ss = fmaf(a0.y, a0.y, ss);
      ss = fmaf(a0.z, a0.z, ss); ss = fmaf(a0.w, a0.w, ss);
      ss = fmaf(a1.x, a1.x, ss); ss = fmaf(a1.y, a1.y, ss);
      ss = fmaf(a1.z, a1.z, ss); ss = fmaf(a1.w, a1.w, ss);
    }
  }
  if (MODE == 2 && xn) {
    ss = warp_sum(ss);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) s_red[warp] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kCombThreads / 32; ++w) tot += s_red[w];
    const float inv_rms = 1.f / sqrtf(tot / (float)d + eps);
    for (int c = threadIdx.x; c < d8; c += kCombThreads) {
      const size_t o = (size_t)t * d + (size_t)c * 8;
      const float4 a0 = reinterpret_cast<const float4*>(x + o)[0];
      const float4 a1 = reinterpret_cast<const float4*>(x + o)[1];
      __nv_bfloat162 b[4] = {__floats2bfloat162_rn(a0.x * inv_rms, a0.y * inv_rms),
                             __floats2bfloat162_rn(a0.z * inv_rms, a0.w * inv_rms),
                             __floats2bfloat162_rn(a1.x * inv_rms, a1.y * inv_rms),
                             __floats2bfloat162_rn(a1.z * inv_rms, a1.w * inv_rms)};
      *reinterpret_cast<uint4*>(xn + o) = *reinterpret_cast<const uint4*>(b);
    }
  }
}

cudaError_t launch_combine(const GemmArgs& a, void* y, bool y_f32, float* x, void* xn, float eps,
                           cudaStream_t s) {
  const int P = a.T * a.k;
  const __half* O = static_cast<const __half*>(a.O);
  __nv_bfloat16* xnb = static_cast<__nv_bfloat16*>(xn);
  prof_begin(K_FINALIZE, s);
  cudaError_t err;
  if (x)
    err = launch_pdl(combine_kernel<2>, dim3(a.T), dim3(kCombThreads), 0, s, O, a.inv,
                     a.gates, a.k, P, a.d, (void*)nullptr, x, xnb, eps, a.status);
  else if (y_f32)
    err = launch_pdl(combine_kernel<0>, dim3(a.T), dim3(kCombThreads), 0, s, O, a.inv,
                     a.gates, a.k, P, a.d, y, (float*)nullptr, (__nv_bfloat16*)nullptr, eps, a.status);
  else
    err = launch_pdl(combine_kernel<1>, dim3(a.T), dim3(kCombThreads), 0, s, O, a.inv,
                     a.gates, a.k, P, a.d, y, (float*)nullptr, (__nv_bfloat16*)nullptr, eps, a.status);
  prof_end(K_FINALIZE, s);
  return err;
}

}  // namespace lily
