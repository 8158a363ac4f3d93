// chunk.cuh -- the chunk-parallel tensor-core kernel for bf16 inputs
// (sm_103a: TMA + tcgen05 + TMEM), instantiated per head size in
// chunk_d64.cu / chunk_d128.cu.
//
// Causal form per chunk of C = 64 tokens (Keras request, "Mathematical
// definition / Causal"; ONNX LinearAttention "may be implemented using
// chunk-parallel algorithms"), written transposed so that the value
// dimension is the MMA's M (= Dv) and the state never leaves tensor memory:
//
//   Y^T   = S_prev^T . phi(Q)^T                    (inter-chunk read-out)
//         + V^T . mask(phi(Q) phi(K)^T)^T          (intra-chunk, j <= i)
//   den_i = phi(q_i).Z_prev + sum_{j<=i} phi(q_i).phi(k_j) + eps
//   S^T  += V^T . phi(K)                           (state carry, fp32)
//   Z    += sum_j phi(k_j)
//
// Gated rule (ONNX "gated", per-head scalar log decay g): with G_i the
// inclusive cumulative sum of g inside the chunk, the read-out uses
// exp(G_i) q_i against S_prev, the intra weights are multiplied by
// exp(G_i - G_j) (<= 1), and the carry is S <- exp(G_C) S + sum_j
// exp(G_C - G_j) k_j v_j^T.
//
// Precision: phi(Q) and phi(K) enter the score product as bf16; the masked
// score matrix is split into bf16 hi + lo parts (~16 significant bits); the
// read-out with the carried state uses the fp32 state in tensor memory
// directly at tf32 precision (linear rule) or a bf16 hi + lo copy of it
// (gated rule, whose state is rescaled every chunk); the state update uses a
// hi + lo split of the key operand whenever phi(k) (or the decayed key) is
// not exactly representable in bf16.  All accumulation is fp32 in tensor
// memory.
//
// Roles (480 threads): warp 0 TMA producer, warp 1 MMA issuer and TMEM
// owner, warps 2-5 state and output (start and final state, the output stage;
// gated rule: also the hi/lo copy of the carried state and its decay), warps
// 6-9 epilogue (masking of the scores, 1/den), warps 10-13 feature maps (phi
// of keys and queries, Z rows and sums), warp 14 (linear causal rule only)
// second MMA issuer: the read-outs with the carried state and the state
// updates, while warp 1 issues the scores and intra products.  Every wait is
// bounded and reports a code in *err instead of hanging.
//
// Pipeline per chunk i (G query heads per kv head): the feature warps run
// ahead of the tensor core, limited only by the load rings; the MMA issues
// per head the scores and the read-out with S_prev, after the last head's
// read-out the state update, then the intra term.  Linear rule: the only
// loop-carried chain is read-out(i) -> update(i) -> read-out(i+1), ordered by
// the MMA issuer alone; gated rule: state hi/lo(i) -> read-out(i) ->
// update(i) -> state hi/lo(i+1) through the state warps.
//
// Modes: kCausal (outputs + carried state), kState (only the state update
// over a segment, for the two-pass sequence split and the non-causal
// reduction), kApply (non-causal read-out with a fixed global state).
#pragma once

#include "chunk_args.h"
#include "common.cuh"
#include "umma.cuh"

namespace la {
namespace chunk {

using namespace umma;

constexpr int kC = 64;  // tokens per chunk
// Per-stage decay block of the gated rule (floats).  G_j is the inclusive
// cumulative log decay inside the chunk.  A step whose log decay is at most
// kRestartLogDecay (a -inf "forget everything" step, taken as kMinLogDecay)
// starts a new group: every weight exp(G_i - G_j) across it is zero in
// float32.  Each group has a reference ref_g in the middle of its G range.
// When every group's range is moderate (the "exact" chunks: spread below 60,
// top below 30) the chunk's read-out takes undecayed queries: the state warps
// hand the tensor core a hi/lo copy of exp(ref_0) S, the intra weights are
// exp(ref_g(j) - G_j) (column factors; zero across groups) and output row i is
// multiplied by exp(G_i - ref_g(i)), so no decayed operand is rounded to
// bf16.  Rows after the first restart read nothing of S (their query rows in
// the read-out copy are zero).  Other chunks take the decayed queries
// exp(G_i) q in bf16 and per-element weights exp(G_i - G_j).
//   [0, 64)   exact: exp(G_i - ref_g(i)) (output factors); else G_i
//   [64, 128) exact: exp(ref_g(j) - G_j) (column factors of the intra weights)
//   kGRef ref_0, kGRefLast ref of the last group, kGTot the chunk's total log
//   decay, kGWord0/1 the 64-bit word of restart steps (bit patterns),
//   kGFlag 0 (not exact), 1 (exact, one group), 2 (exact, several groups)
constexpr int kGCol = 64, kGRef = 128, kGFlag = 129, kGTot = 130, kGRefLast = 131, kGWord0 = 132, kGWord1 = 133;
// Floor of a step's log decay (gated rule).  exp(-200) underflows to zero in
// float32 (the smallest subnormal is ~exp(-103.3)), so a step at the floor
// erases the earlier state exactly as -inf does, as long as the later steps
// of its 64-token chunk do not add up to more than +97 (log decays are
// log-sigmoid values, <= 0, in every workload of the pages).
constexpr float kMinLogDecay = -200.f;
// A step with a log decay at or below this starts a new group of its chunk
// (see the decay block): exp(-100) is below float32's smallest normal number.
constexpr float kRestartLogDecay = -100.f;

// Restart steps of a chunk as a 64-bit word (bit j = step j) from the
// per-lane flags of steps 2 lane (even) and 2 lane + 1 (odd); warp-collective.
__device__ __forceinline__ uint64_t restart_word(bool even, bool odd) {
    auto spread = [](uint64_t x) {  // bit i -> bit 2i
        x = (x | (x << 16)) & 0x0000FFFF0000FFFFull;
        x = (x | (x << 8)) & 0x00FF00FF00FF00FFull;
        x = (x | (x << 4)) & 0x0F0F0F0F0F0F0F0Full;
        x = (x | (x << 2)) & 0x3333333333333333ull;
        x = (x | (x << 1)) & 0x5555555555555555ull;
        return x;
    };
    const uint32_t e = __ballot_sync(0xffffffffu, even), o = __ballot_sync(0xffffffffu, odd);
    return spread(e) | (spread(o) << 1);
}
// No restart step in (j, i] (0 <= j <= i <= 63): steps j and i are in one group.
__device__ __forceinline__ bool same_group(uint64_t word, int j, int i) {
    if (i == j) return true;
    const uint64_t span = (i - j == 64) ? ~0ull : ((1ull << (i - j)) - 1);
    return ((word >> (j + 1)) & span) == 0;
}
__device__ __forceinline__ uint64_t gc_word(const float* gc) {
    return (uint64_t)__float_as_uint(gc[kGWord0]) | ((uint64_t)__float_as_uint(gc[kGWord1]) << 32);
}
constexpr int kThreads = 480;  // 15 warps; the two-issuer kernel adds warp 15
template <bool SPLIT>
constexpr int block_threads() { return SPLIT ? 512 : kThreads; }
constexpr int kStateWarp0 = 2, kEpiWarp0 = 6, kFeatWarp0 = 10, kMmaSWarp = 14;  // warp 15: see kFeatMovedTo

// AT2: two masked-score buffers where shared memory holds them (the
// two-issuer kernel for grouped query heads)
template <int D, int MODE, bool NORM, int FMAP, bool GATED, bool OUT_BF16, bool AT2 = false>
struct Cfg {
    // the state update takes its key operand as bf16 hi + lo wherever that
    // operand is not exactly a bf16 value: the gated rule's decayed keys, and
    // phi(k) of elu+1 (x + 1 or exp(x); rounded to bf16 alone it would carry
    // up to 2^-8 of relative error into every state row).  relu + eps of a bf16
    // input rounds back to the input (eps is far below its ulp) and the
    // identity map is exact, so those keys enter as one bf16 part.
    static constexpr bool kSplitK = GATED || FMAP == LA_FMAP_ELU_PLUS_ONE;
    static constexpr bool kHasKV = MODE != kApply;
    static constexpr bool kHasQ = MODE != kState;
    static constexpr int kTile = D * 128;  // 64 rows x D bf16 (D/64 swizzled blocks of 8 KB)
    static constexpr int kZr = D * 16;     // 8 rows x D bf16: [Z_hi; Z_lo; 0 x 6]
    // key tile: per 64-feature block, 64 token rows followed (causal with the
    // normalizer) by 8 Z rows, so one N = 72 MMA gives the scores and phi(q).Z
    static constexpr int kKRows = (NORM && MODE == kCausal) ? 72 : 64;
    static constexpr int kKBlk = kKRows * 128;  // bytes per 64-feature block of the key tile
    static constexpr int kKTile = (D / 64) * kKBlk;
    // per KV stage: Kb (+ Z rows) | Kd (gated) | Klo (split) | Vb; the gated
    // rule's decay block of each stage lives after the barriers (kGStage)
    static constexpr int kOffKd = ((kKTile + 1023) / 1024) * 1024;
    static constexpr int kOffKlo = kOffKd + (GATED ? kTile : 0);
    static constexpr int kOffVb = kOffKlo + (kSplitK ? kTile : 0);
    static constexpr int kOffG = kOffVb + kTile;
    static constexpr int kKvStage = kHasKV ? kOffG : 0;
    // gated rule: the chunk's decay block (cumulative log decay, factored
    // weights, reference, flag: 130 floats, 544 bytes) of each key/value stage,
    // kept after the barriers so that the stages stay multiples of 1 KB
    static constexpr int kGFloats = 136;
    static constexpr int kGStage = (GATED && kHasKV) ? kGFloats * 4 : 0;
    // linear rule: the read-out with the carried state runs as kind::tf32
    // with the fp32 state straight from TMEM as A, against an fp32 copy of
    // phi(Q) (64 x D, D/32 swizzled blocks of 8 KB); the gated rule, whose
    // state is rescaled every chunk anyway, reads a bf16 hi/lo copy of it
    static constexpr bool kTf32 = !GATED;
    // linear causal with grouped query heads (G > 1) or at head size 128
    // (decided at launch): two MMA issuers -- warp 1 the scores and the intra
    // products, warp 14 the read-outs of all G heads with the carried state
    // and the state updates -- so that the waits of one overlap the issue of
    // the other.  At head size 64 with one query head per kv head the single
    // issuer interleaves them better.
    static constexpr bool kSplitMma = kTf32 && MODE == kCausal;
    static constexpr int kQf = (kHasQ && kTf32) ? 2 * kTile : 0;
    static constexpr int kQStage = kHasQ ? kTile * (GATED ? 2 : 1) + kQf : 0;
    // masked scores as bf16 hi + lo (~16 significant bits): one bf16 part
    // would put up to 2^-9 of relative error on single output rows (the first
    // token of a sequence is one score times one value row)
    static constexpr bool kALo = true;
    // masked-score buffers (hi, lo: 64 x 64 bf16 each): the epilogue writes
    // item n's once the intra product of item n - kNAT has completed; two when
    // shared memory holds them at the ring depths one buffer allows (below)
    static constexpr int kZrApply = (MODE == kApply && NORM) ? kZr : 0;
    // bf16 output: each item's 64 x D output tile is staged in shared memory
    // and leaves with 16-byte stores.  Row pitch D + 8 elements (16 bytes of
    // padding against bank conflicts of the head-size-64 transposed writes);
    // the gated rule at head size 128, whose writes are 64 contiguous bytes
    // per warp, uses the unpadded pitch to fit its budget
    static constexpr bool kYStage = OUT_BF16 && MODE != kState;
    static constexpr int kYPitch = (GATED && D == 128) ? D : D + 8;
    static constexpr int kYS = kYStage ? 64 * kYPitch * 2 : 0;
    // feature-map warps: 4 (warps 10-13), or 8 in the state pass (warps 6-13),
    // which has no scores for the epilogue warps to mask
    static constexpr int kFeatWarps = MODE == kState ? 8 : 4;
    static constexpr int kFeatW0 = MODE == kState ? kEpiWarp0 : kFeatWarp0;
    static constexpr int kFeatThreads = 32 * kFeatWarps;
    // vectorised tile passes of the feature warps: 16-byte chunks
    static constexpr int kCPR = D / 8;                    // chunks per 64 x D tile row
    static constexpr int kRowStep = kFeatThreads / kCPR;  // rows covered by one pass
    static constexpr int kPer = 64 / kRowStep;            // chunks per thread per tile
    static_assert(kRowStep * kPer == 64, "feature pass covers the tile");
    static constexpr int kZpart = kRowStep * D;  // floats of one buffer of partial Z sums
    // 1/den ring and partial Z sums (x2) -- the normalizer's, so not for the
    // gated rule, which has none -- then the barriers
    static constexpr int kMiscNorm = GATED ? 0 : 1024 + 2 * kZpart * 4;
    static constexpr int kMisc = kMiscNorm + 512;
    static constexpr int bytes(int nkv, int nq, int nat = MODE == kCausal ? 1 : 0) {
        return 1024 + nkv * kKvStage + nq * kQStage + nat * 2 * 8192 + kZrApply + kYS + kMisc + nkv * kGStage;
    }
    // the linear rule's state pass at head size 64 runs two CTAs per SM (its
    // ring sized for half the shared memory, its TMEM the state's D
    // columns): the two-pass sequence split then runs its state pass on twice
    // as many, half-length sub-segments in one wave.  (The gated state pass
    // would spill at the register budget of two CTAs.)
    static constexpr bool kTwoPerSm = MODE == kState && D == 64 && !GATED;
    static constexpr int kLimit = kTwoPerSm ? 113 * 1024 : 227 * 1024;
    // ring depths: the deepest of (4,4), (4,3), (3,3), (3,2), (2,2) that
    // shared memory holds (key/value and query stages), else fewer
    static constexpr bool fits(int nkv, int nq) {
        return bytes(kHasKV ? nkv : 0, kHasQ ? nq : 0) <= kLimit;
    }
    static constexpr int kNKV0 = fits(4, 4) ? 4 : fits(4, 3) ? 4 : fits(3, 3) ? 3 : fits(3, 2) ? 3 : fits(2, 2) ? 2
                                 : fits(2, 1) ? 2 : 1;
    static constexpr int kNQ0 = fits(kNKV0, 4) ? 4 : fits(kNKV0, 3) ? 3 : fits(kNKV0, 2) ? 2 : 1;
    static constexpr int kNKV = kHasKV ? kNKV0 : 0;
    static constexpr int kNQ = kHasQ ? kNQ0 : 0;
    static constexpr int kNAT = MODE != kCausal ? 0 : (AT2 && bytes(kNKV, kNQ, 2) <= kLimit) ? 2 : 1;
    static constexpr int kAT = kNAT * 2 * 8192;
    static_assert(kNKV <= 4 && kNQ <= 4, "barrier arrays hold four stages");
    static constexpr int kSmem = bytes(kNKV, kNQ, kNAT);
    static_assert(kSmem <= kLimit, "shared memory budget");
    // TMEM columns
    // score buffers (64 + 8 columns for phi(q).Z each); the linear rule needs
    // no bf16 copy of the state, so its two buffers take those columns
    static constexpr int kNA = (D == 64 || kTf32) ? 2 : 1;
    static constexpr int kNY = 2;                  // Y^T buffers (64 columns each)
    static constexpr uint32_t kColS = 0;           // S^T fp32: D columns, lanes = value rows
    static constexpr uint32_t kColHi = D;          // S^T hi bf16 pairs: D/2 columns (gated)
    static constexpr uint32_t kColLo = D + D / 2;  // S^T lo (gated)
    static constexpr uint32_t kColA = kTf32 ? D : 2 * D;  // score buffers, 80 columns apart
    static constexpr uint32_t kColY = kColA + 80 * kNA;
    static constexpr uint32_t kTmemCols = MODE == kState ? D : 512;  // the state pass holds S^T alone
    static_assert(MODE == kState || kColY + 64 * kNY <= kTmemCols, "TMEM budget");
};

// Rounds a shared-memory pointer up to 1024 bytes by pointer arithmetic (not
// through an integer), so the compiler still knows it addresses shared memory
// and emits shared loads/stores instead of generic ones.
template <bool B>
struct BoolTag {
    static constexpr bool value = B;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return p + ((1024u - (smem_u32(p) & 1023u)) & 1023u);
}

__device__ __forceinline__ void bf8_to_f(const uint4& u, float (&f)[8]) {
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 t = __bfloat1622float2(p[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}
__device__ __forceinline__ uint32_t bf2_bits(__nv_bfloat162 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ uint4 f_to_bf8(const float (&f)[8]) {
    return make_uint4(bf2_bits(__floats2bfloat162_rn(f[0], f[1])), bf2_bits(__floats2bfloat162_rn(f[2], f[3])),
                      bf2_bits(__floats2bfloat162_rn(f[4], f[5])), bf2_bits(__floats2bfloat162_rn(f[6], f[7])));
}
// x = hi + lo with hi = bf16(x) and lo = bf16(x - hi), for a pair
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(h);
    hi = bf2_bits(h);
    lo = bf2_bits(__floats2bfloat162_rn(x0 - hf.x, x1 - hf.y));
}
__device__ __forceinline__ void split8(const float (&f)[8], uint4& hi, uint4& lo) {
    split2(f[0], f[1], hi.x, lo.x);
    split2(f[2], f[3], hi.y, lo.y);
    split2(f[4], f[5], hi.z, lo.z);
    split2(f[6], f[7], hi.w, lo.w);
}
__device__ __forceinline__ __nv_bfloat16& bf_at(uint8_t* base, uint32_t off) {
    return *reinterpret_cast<__nv_bfloat16*>(base + off);
}

// SPLIT: 0 one MMA issuer; 1 two MMA issuers (linear causal rule at head
// size 128 with one query head per kv head); 2 two MMA issuers for grouped
// query heads, with two masked-score buffers where they fit and the scores of
// the next item issued ahead of the current intra product (see
// Cfg::kSplitMma).  Separate instantiations, so that each kernel carries only
// the issue code it runs.  MASK: the sequence-validity
// mask is read (Keras request, Masking); without it the mask pointer is a
// constant null and every mask branch folds away, so unmasked calls run
// exactly the code they would run without mask support.
template <int D, int MODE, bool NORM, int FMAP, bool GATED, bool OUT_BF16, int SPLIT = 0, bool MASK = false>
__global__ void __launch_bounds__(block_threads<Cfg<D, MODE, NORM, FMAP, GATED, OUT_BF16>::kSplitMma && SPLIT != 0>(),
                                  Cfg<D, MODE, NORM, FMAP, GATED, OUT_BF16>::kTwoPerSm ? 2 : 1)
    chunk_kernel(const __grid_constant__ Args a, const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
                 const __grid_constant__ CUtensorMap mapV) {
    using Cf = Cfg<D, MODE, NORM, FMAP, GATED, OUT_BF16, SPLIT == 2>;
    constexpr bool SPLITK = Cf::kSplitK;
    constexpr bool TF32 = Cf::kTf32;
    constexpr bool ALO = Cf::kALo;
    constexpr int NA = Cf::kNA, NY = Cf::kNY;
    constexpr int NKV = Cf::kNKV, NQ = Cf::kNQ;
    constexpr int NKV1 = NKV ? NKV : 1, NQ1 = NQ ? NQ : 1;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    uint8_t* kv_base = sm;
    uint8_t* q_base = kv_base + NKV * Cf::kKvStage;
    uint8_t* at_base = q_base + NQ * Cf::kQStage;
    uint8_t* zr_apply = at_base + Cf::kAT;
    uint8_t* ystage = zr_apply + Cf::kZrApply;  // staged output tile (64 x D bf16)
    float* misc = reinterpret_cast<float*>(ystage + Cf::kYS);
    float* inv_den = misc;           // [4][64] scale / den of the last four items (normalizer)
    float* zpart = misc + 256;       // [2][kZpart] partial column sums of phi(K) (normalizer)
    uint64_t* bars = reinterpret_cast<uint64_t*>(misc + Cf::kMiscNorm / 4);
    float* garea = reinterpret_cast<float*>(bars + 64);  // gated: [NKV][kGFloats] decay blocks
    uint64_t* full_kv = bars;        // [4] ring stages
    uint64_t* empty_kv = bars + 4;   // [4]
    uint64_t* conv_kv = bars + 8;    // [4]
    uint64_t* full_q = bars + 12;    // [4]
    uint64_t* empty_q = bars + 16;   // [4]
    uint64_t* conv_q = bars + 20;    // [4]
    uint64_t* a_full = bars + 24;    // [2]
    uint64_t* a_empty = bars + 26;   // [2]
    uint64_t* at_full = bars + 28;   // [2] masked scores written (per buffer)
    uint64_t* y_full = bars + 32;    // [2]
    uint64_t* y_empty = bars + 34;   // [2]
    uint64_t* state_ready = bars + 36;
    uint64_t* state_done = bars + 37;
    uint64_t* conv_group = bars + 38;  // barrier among the feature warps
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 39);
    uint64_t* inter_done = bars + 40;  // tf32 read-outs of a chunk complete (state may be updated)
    uint64_t* final_done = bars + 41;  // every tensor-core operation of the CTA complete
    // [4] scale/den of item n in inv_den[n & 3] (normalizer only).  Four
    // phases in flight at most: the scores of item n + 4 are issued only
    // after the output stage has read item n + 1 out of TMEM.
    uint64_t* den_full = bars + 42;  // [4]
    uint64_t* inter_cmp = bars + 50;  // [2] read-out of item n complete (split issue; per Y^T buffer)
    uint64_t* upd_done = bars + 52;   // state update of a chunk complete (split issue)
    uint64_t* out_group = bars + 55;  // barrier among the four output warps (staged output tile)
    uint32_t ophase = 0;              // this thread's uses of out_group

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bh = blockIdx.x;
    const int seg = blockIdx.y;
    // Argument fields in registers: the role code below runs in lambdas that
    // capture by reference, and reading the parameter block through its
    // address inside hot loops would be a long-latency load per use.
    const int T = a.T, Hq = a.Hq, Hkv = a.Hkv, G = a.G, nseg = a.nseg;
    constexpr bool split = Cf::kSplitMma && SPLIT != 0;  // two MMA issuers
    constexpr int fmap = FMAP;
    const float eps = a.eps, scale = a.scale;
    const __nv_bfloat16* __restrict__ decay = a.decay;
    const uint8_t* __restrict__ mask = MASK ? a.mask : nullptr;
    void* const yout = a.y;
    const int b = bh / Hkv, hk = bh - b * Hkv;
    const int nchunks = (T + kC - 1) / kC;
    const int c_begin = seg * a.cps;
    const int nck = min(nchunks, c_begin + a.cps) - c_begin;
    // Validity of the steps t0 .. t0 + 63 of this sequence as a 64-bit word
    // (Keras request, Masking; steps past T count as valid, they are cut
    // elsewhere).  Warp-collective: two loads per lane and two ballots.
    // The mask bytes of steps t0 + lane and t0 + 32 + lane (1 past the end),
    // loaded ahead of use; valid_bits turns them into the word.
    auto mask_bytes = [&](int t0) -> uint32_t {
        if (!mask) return 0x101u;
        const size_t bt = (size_t)b * T + t0;
        const uint32_t m0 = t0 + lane >= T ? 1u : mask[bt + lane];
        const uint32_t m1 = t0 + 32 + lane >= T ? 1u : mask[bt + 32 + lane];
        return (m0 != 0) | ((m1 != 0) << 8);
    };
    auto valid_bits = [&](uint32_t mb) -> uint64_t {
        if (!mask) return ~0ull;
        return (uint64_t)__ballot_sync(0xffffffffu, mb & 0xffu) | ((uint64_t)__ballot_sync(0xffffffffu, mb >> 8) << 32);
    };
    auto valid_word = [&](int t0) -> uint64_t { return valid_bits(mask_bytes(t0)); };

    auto Kb = [&](int s) { return kv_base + s * Cf::kKvStage; };
    auto Kd = [&](int s) { return kv_base + s * Cf::kKvStage + Cf::kOffKd; };
    auto Klo = [&](int s) { return kv_base + s * Cf::kKvStage + Cf::kOffKlo; };
    auto Vb = [&](int s) { return kv_base + s * Cf::kKvStage + Cf::kOffVb; };
    // Z rows [Z_hi; Z_lo; 0 x 6]: behind the key rows of each 64-feature block
    // (causal), or one standalone 8-row block per feature block (read-out pass)
    auto zr_at = [&](int s, int kb) -> uint8_t* {
        return MODE == kApply ? zr_apply + kb * 1024 : kv_base + s * Cf::kKvStage + kb * Cf::kKBlk + 64 * 128;
    };
    auto Gc = [&](int s) { return garea + s * Cf::kGFloats; };
    auto Qb = [&](int s) { return q_base + s * Cf::kQStage; };
    auto Qd = [&](int s) { return q_base + s * Cf::kQStage + Cf::kTile; };
    auto Qf = [&](int s) { return q_base + s * Cf::kQStage + Cf::kTile; };  // fp32 phi(Q) (linear rule)
    constexpr int NAT = Cf::kNAT ? Cf::kNAT : 1;
    auto ATh = [&](int buf) { return at_base + buf * 16384; };  // masked scores, hi part
    auto ATl = [&](int buf) { return at_base + buf * 16384 + 8192; };  // lo part

    if (tid == 0) {
        for (int i = 0; i < 4; ++i) {
            mbar_init(&full_kv[i], 1);
            mbar_init(&empty_kv[i], split ? 2 : 1);
            mbar_init(&conv_kv[i], Cf::kFeatWarps);
            mbar_init(&full_q[i], 1);
            mbar_init(&empty_q[i], split ? 2 : 1);
            mbar_init(&conv_q[i], Cf::kFeatWarps);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&a_full[i], 1);
            mbar_init(&a_empty[i], 4);
            mbar_init(&at_full[i], 4);
            mbar_init(&y_full[i], 1);
            mbar_init(&y_empty[i], 4);
        }
        mbar_init(state_ready, 4);
        mbar_init(state_done, 1);
        mbar_init(conv_group, Cf::kFeatWarps);
        for (int i = 0; i < 4; ++i) mbar_init(&den_full[i], 4);
        mbar_init(inter_done, 1);
        mbar_init(final_done, split ? 2 : 1);
        for (int i = 0; i < 2; ++i) mbar_init(&inter_cmp[i], 1);
        mbar_init(upd_done, 1);
        mbar_init(out_group, 4);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, Cf::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        if (Cf::kHasQ) tma_prefetch(&mapQ);
        if (Cf::kHasKV) {
            tma_prefetch(&mapK);
            tma_prefetch(&mapV);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // state pass: the causal pass that consumes its increments may launch now
    // (programmatic dependent launch); it waits for this grid's completion
    // only where it reads them
    if (MODE == kState && tid == 0) griddep_launch_dependents();
    const uint32_t tmem = *tmem_slot;
    unsigned* err = a.err;

    // Query head item n (chunk i): feature map in place (bf16), plus the fp32
    // copy for the tf32 read-out, or the decayed copy of the gated rule.  Run
    // by 128 threads (qt = 0..127, whole warps): the feature warps, or, for the
    // linear causal kernel with one query head per kv head, the epilogue
    // warps, which convert item n + 1 right after masking the scores of item n
    // and so take this work off the feature warps that pace the keys.
    auto q_features = [&](int i, int n, int qt) -> bool {
        constexpr int kCPR = Cf::kCPR, kRowStep = Cf::kRowStep, kPer = Cf::kPer;
        const int cc = qt % kCPR, rbase = qt / kCPR;
        auto chunk_off = [&](int m) -> uint32_t {
            const int row = rbase + kRowStep * m;
            return static_cast<uint32_t>((cc >> 3) * 8192 + row * 128 + ((((cc & 7) ^ (row & 7))) << 4));
        };
        const int sq = n % NQ1;
        if (!warp_wait(&full_q[sq], (n / NQ1) & 1, err, kErrFullQ)) return false;
        // gated rule, exact chunk of one group: the read-out takes the queries
        // as they are; with restarts it takes a copy whose rows after the
        // first restart are zero
        const float qflag = GATED ? Gc(i % NKV1)[kGFlag] : 0.f;
        if ((fmap != LA_FMAP_NONE || GATED || TF32) && qflag != 1.f) {
            const float* gc = Gc(i % NKV1);
            const uint64_t qword = qflag == 2.f ? gc_word(gc) : 0ull;
            uint4 nxt = *reinterpret_cast<const uint4*>(Qb(sq) + chunk_off(0));
#pragma unroll 1
            for (int m = 0; m < kPer; ++m) {
                const uint4 cur = nxt;
                if (m + 1 < kPer) nxt = *reinterpret_cast<const uint4*>(Qb(sq) + chunk_off(m + 1));
                float f[8];
                bf8_to_f(cur, f);
                if (GATED) {
                    const int row = rbase + kRowStep * m;
                    const float w = qflag == 2.f ? (same_group(qword, 0, row) && !(qword & 1ull) ? 1.f : 0.f)
                                                 : __expf(gc[row]);
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] *= w;
                    *reinterpret_cast<uint4*>(Qd(sq) + chunk_off(m)) = f_to_bf8(f);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = phi<true>(fmap, f[e], eps);
                    if (fmap != LA_FMAP_NONE) *reinterpret_cast<uint4*>(Qb(sq) + chunk_off(m)) = f_to_bf8(f);
                    if (TF32) {
                        // features 8cc..8cc+7 are two 16-byte chunks of a 32-feature block
                        const int row = rbase + kRowStep * m;
                        uint8_t* blk = Qf(sq) + (cc >> 2) * 8192 + row * 128;
                        const int c16 = 2 * (cc & 3);
                        *reinterpret_cast<float4*>(blk + ((c16 ^ (row & 7)) << 4)) =
                            make_float4(f[0], f[1], f[2], f[3]);
                        *reinterpret_cast<float4*>(blk + (((c16 + 1) ^ (row & 7)) << 4)) =
                            make_float4(f[4], f[5], f[6], f[7]);
                    }
                }
            }
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(&conv_q[sq]);
        return true;
    };
    constexpr bool kQOnEpi = MODE == kCausal && !GATED && !split;
    // Warp w runs on sub-partition w % 4.  In the causal pass, feature warp
    // slot 3 (warp 13) would share the MMA warp's sub-partition (that of warp
    // 1) with two other busy warps, so it moves: to warp 14 when there is no
    // second MMA issuer, else to warp 15 (the feature warps use no TMEM lanes
    // and may run anywhere).  Warp 13, and the warps no role claims, idle.
    constexpr bool kFeatMove = MODE == kCausal;
    constexpr int kFeatMovedTo = split ? 15 : 14;
    constexpr int kIdleWarp = (MODE == kCausal && !split) ? 13 : kMmaSWarp;  // or the second issuer

    // Output of item m (query head m % G of chunk m / G): Y^T from TMEM times
    // scale/den, stored to global memory.  Run by four warps, one per TMEM lane
    // quadrant: the state warps (linear rule) or the epilogue warps (gated).
    // gated rule, exact chunk (gexact): output row x is also multiplied by
    // exp(G_x - ref), lane l of the warp holding that factor for rows l (eo_lo)
    // and l + 32 (eo_hi); tok_f(x) gives row x's whole factor (warp-collective)
    auto emit_y = [&](int m, float eo_lo = 1.f, float eo_hi = 1.f, bool gexact = false) -> bool {
        auto tok_f = [&](int x) -> float {
            if constexpr (GATED) {
                const float e = __shfl_sync(0xffffffffu, x < 32 ? eo_lo : eo_hi, x & 31);
                return gexact ? scale * e : scale;
            } else {
                return scale;
            }
        };
        const int quad = warp & 3;
        const bool m64 = D == 64;
        const int vrow = m64 ? (quad * 16 + lane) : (quad * 32 + lane);  // value index of this Y^T lane
        const bool vrow_ok = m64 ? lane < 16 : true;
        const int i_chunk = m / G, r_head = m - i_chunk * G;
        const int t0 = (c_begin + i_chunk) * kC;
        const int valid = min(kC, T - t0);
        const int yb = m % NY;
        if (!warp_wait(&y_full[yb], (m / NY) & 1, err, kErrYFull)) return false;
        tc_fence_after();
        const uint64_t okw = valid_word(t0);  // invalid steps get zero output rows
        // all 64 tokens of this lane in one round trip to TMEM; the buffer is
        // released before the stores.  Head size 64 with a staged tile: Y^T is
        // an M = 64 tile (lanes 0-15 of each quadrant), read in the 16x256b
        // shape so that all 32 lanes work (y0 then holds value rows
        // 16 quad + lane/4 and + 8, tokens 8g + 2(lane%4) and + 1).
        constexpr bool kHalfLanes = Cf::kYStage && D == 64;
        uint32_t y0[32], y1[32];
        if constexpr (kHalfLanes) {
            tmem_ld16x256b_x8(tmem_addr(tmem + Cf::kColY + 64 * yb, quad * 32, 0), y0);
        } else {
            tmem_ld32(tmem_addr(tmem + Cf::kColY + 64 * yb, quad * 32, 0), y0);
            tmem_ld32(tmem_addr(tmem + Cf::kColY + 64 * yb, quad * 32, 32), y1);
        }
        tmem_ld_wait();
        reg_fence(y0);
        if constexpr (!kHalfLanes) reg_fence(y1);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&y_empty[yb]);
        // scale/den of item m, written by the four score warps
        if (NORM && !warp_wait(&den_full[m & 3], (m >> 2) & 1, err, kErrYFull)) return false;
        const float4* idn4 = reinterpret_cast<const float4*>(inv_den + (m & 3) * 64);
        const size_t tstride = (size_t)Hq * D;
        const size_t base = (((size_t)b * T + t0) * Hq + hk * G + r_head) * D + vrow;
        if constexpr (Cf::kYStage) {
            // tile [token][D] in shared memory, then 16-byte stores of its valid
            // rows by the four output warps (bounded group barrier)
            __nv_bfloat16* ys = reinterpret_cast<__nv_bfloat16*>(ystage);
            constexpr int P = Cf::kYPitch;
            if constexpr (kHalfLanes) {
                const int v1 = quad * 16 + (lane >> 2), v2 = v1 + 8, cq = 2 * (lane & 3);
                const float* idn = inv_den + (m & 3) * 64;
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    const int x = 8 * g + cq;
                    const float2 f = NORM ? *reinterpret_cast<const float2*>(idn + x) : make_float2(tok_f(x), tok_f(x + 1));
                    ys[x * P + v1] = __float2bfloat16_rn(f.x * __uint_as_float(y0[4 * g]));
                    ys[(x + 1) * P + v1] = __float2bfloat16_rn(f.y * __uint_as_float(y0[4 * g + 1]));
                    ys[x * P + v2] = __float2bfloat16_rn(f.x * __uint_as_float(y0[4 * g + 2]));
                    ys[(x + 1) * P + v2] = __float2bfloat16_rn(f.y * __uint_as_float(y0[4 * g + 3]));
                }
            } else {
                static_assert(D == 128, "the staged 32-lane path covers head size 128 (every lane a value row)");
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    float f[8];
                    if constexpr (NORM) {
                        const float4 fa = idn4[2 * g], fb = idn4[2 * g + 1];
                        f[0] = fa.x, f[1] = fa.y, f[2] = fa.z, f[3] = fa.w, f[4] = fb.x, f[5] = fb.y, f[6] = fb.z,
                        f[7] = fb.w;
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) f[e] = tok_f(g * 8 + e);
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int x = g * 8 + e;
                        ys[x * P + vrow] = __float2bfloat16_rn(f[e] * __uint_as_float(x < 32 ? y0[x] : y1[x - 32]));
                    }
                }
            }
            if (!group_sync(out_group, ophase, err, kErrYFull)) return false;
            const int ot = tid - kStateWarp0 * 32;  // 0..127
            constexpr int kCpr = D / 8;            // 16-byte chunks per row
            __nv_bfloat16* yrow0 = reinterpret_cast<__nv_bfloat16*>(yout) + (base - vrow);
#pragma unroll
            for (int c = ot; c < 64 * kCpr; c += 128) {
                const int x = c / kCpr, cc = c - x * kCpr;
                if (x < valid)
                    *reinterpret_cast<uint4*>(yrow0 + x * tstride + cc * 8) =
                        (okw >> x) & 1 ? *reinterpret_cast<const uint4*>(ys + x * P + cc * 8) : make_uint4(0, 0, 0, 0);
            }
            if (!group_sync(out_group, ophase, err, kErrYFull)) return false;  // tile free again
        } else {
            // every lane runs the loop (the row factors are warp-collective);
            // lanes without a value row store nothing
#pragma unroll
            for (int g = 0; g < 8; ++g) {
                float f[8];
                if constexpr (NORM) {
                    const float4 fa = idn4[2 * g], fb = idn4[2 * g + 1];
                    f[0] = fa.x, f[1] = fa.y, f[2] = fa.z, f[3] = fa.w, f[4] = fb.x, f[5] = fb.y, f[6] = fb.z,
                    f[7] = fb.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = tok_f(g * 8 + e);
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int x = g * 8 + e;
                    const float o = (okw >> x) & 1 ? f[e] * __uint_as_float(x < 32 ? y0[x] : y1[x - 32]) : 0.f;
                    if (vrow_ok && x < valid) {
                        if (OUT_BF16)
                            reinterpret_cast<__nv_bfloat16*>(yout)[base + x * tstride] = __float2bfloat16_rn(o);
                        else
                            reinterpret_cast<float*>(yout)[base + x * tstride] = o;
                    }
                }
            }
        }
        return true;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // loads in the order the converters consume: K/V of chunk i, then its heads
        if (lane == 0) {
            bool ok = true;
            for (int i = 0; i < nck && ok; ++i) {
                const int t0 = (c_begin + i) * kC;
                if (Cf::kHasKV) {
                    const int s = i % NKV1;
                    if (i >= NKV) ok = mbar_wait(&empty_kv[s], ((i / NKV1) & 1) ^ 1, err, kErrEmptyKV);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&full_kv[s], 2 * Cf::kTile);
                    for (int kb = 0; kb < D / 64; ++kb) {
                        tma_load_4d(Kb(s) + kb * Cf::kKBlk, &mapK, &full_kv[s], kb * 64, hk, t0, b);
                        tma_load_4d(Vb(s) + kb * 8192, &mapV, &full_kv[s], kb * 64, hk, t0, b);
                    }
                }
                if (Cf::kHasQ) {
                    for (int r = 0; r < G && ok; ++r) {
                        const int n = i * G + r, s = n % NQ1;
                        if (n >= NQ) ok = mbar_wait(&empty_q[s], ((n / NQ1) & 1) ^ 1, err, kErrEmptyQ);
                        if (!ok) break;
                        mbar_arrive_expect_tx(&full_q[s], Cf::kTile);
                        for (int kb = 0; kb < D / 64; ++kb)
                            tma_load_4d(Qb(s) + kb * 8192, &mapQ, &full_q[s], kb * 64, hk * G + r, t0, b);
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------- MMA issuer
        // The whole warp runs this loop, so that every operand is warp-uniform
        // (descriptors stay in uniform registers); lane 0 alone issues the
        // tensor-core instructions through their predicate.
        {
            const uint32_t lead = lane == 0;
            bool ok = true;
            constexpr uint32_t id_scores = idesc_bf16(64, Cf::kKRows, false, false);
            constexpr uint32_t id_qz = idesc_bf16(64, 8, false, false);
            constexpr uint32_t id_inter = idesc_bf16(D, 64, false, false);
            constexpr uint32_t id_inter_tf32 = idesc_tf32(D, 64);
            constexpr uint32_t id_intra = idesc_bf16(D, 64, true, false);
            constexpr uint32_t id_state = idesc_bf16(D, D, true, true);
            const uint32_t tS = tmem + Cf::kColS, tHi = tmem + Cf::kColHi, tLo = tmem + Cf::kColLo;
            // the issue loops of the linear rule at head size 128 run unrolled
            // (the tensor core there waits on the issuing warp); the others keep
            // the compact loops, whose smaller code the other roles share
            constexpr int kUnr = (TF32 && D == 128) ? 16 : 1;

            // state update of chunk i: S^T += V^T . Kd (+ V^T . Kd_lo)
            auto issue_state_update = [&](int s) {
                uint8_t* khi = GATED ? Kd(s) : Kb(s);
                const uint32_t khi_lbo = GATED ? 8192u : (uint32_t)Cf::kKBlk;  // stride of 64-feature blocks
                const uint64_t dv0 = sdesc_sw128(smem_u32(Vb(s)), 8192, 1024);
                const uint64_t dk0 = sdesc_sw128(smem_u32(khi), khi_lbo, 1024);
                const uint64_t dl0 = sdesc_sw128(smem_u32(Klo(s)), 8192, 1024);
#pragma unroll kUnr
                for (int ks = 0; ks < kC / 16; ++ks) {
                    const uint64_t o = (uint64_t)(ks * 2048 >> 4);
                    mma_ss(tS, dv0 + o, dk0 + o, id_state, 1, lead);
                    if (SPLITK) mma_ss(tS, dv0 + o, dl0 + o, id_state, 1, lead);
                }
            };

            if constexpr (split) {
                if constexpr (SPLIT == 2) {
                // scores and intra products; the read-outs and updates are warp 14's.
                // Grouped query heads (SPLIT 2): the scores of item n + 1 go out
                // before the intra product of item n, so the epilogue masks them
                // while that product waits for its masked scores; crossing into
                // the next chunk needs a second key/value stage (this warp
                // releases the current one at its end).  With one query head per
                // kv head the look-ahead (which then always crosses into the next
                // chunk) measured slower.
                const int N = nck * G;
                auto issue_scores = [&](int n) -> bool {
                    const int i = n / G, r = n - i * G, s = i % NKV1, sq = n % NQ1, ab = n % NA;
                    if (r == 0) {
                        if (!warp_wait(&conv_kv[s], (i / NKV1) & 1, err, kErrConvKV)) return false;
                        tc_fence_after();
                    }
                    if (!warp_wait(&conv_q[sq], (n / NQ1) & 1, err, kErrConvQ)) return false;
                    tc_fence_after();
                    if (n >= NA) {
                        if (!warp_wait(&a_empty[ab], ((n / NA) & 1) ^ 1, err, kErrAEmpty)) return false;
                        tc_fence_after();
                    }
                    // scores, and in columns 64..71 phi(q).[Z_hi; Z_lo] from the Z rows
                    const uint32_t tA = tmem + Cf::kColA + 80 * ab;
                    const uint64_t dq0 = sdesc_sw128(smem_u32(Qb(sq)), 16, 1024);
                    const uint64_t dk0 = sdesc_sw128(smem_u32(Kb(s)), 16, 1024);
#pragma unroll 1
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t qo = (ks >> 2) * 8192 + (ks & 3) * 32;
                        const uint32_t ko = (ks >> 2) * Cf::kKBlk + (ks & 3) * 32;
                        mma_ss(tA, dq0 + (qo >> 4), dk0 + (ko >> 4), id_scores, ks > 0, lead);
                    }
                    mma_commit(&a_full[ab], lead);
                    mma_commit(&empty_q[sq], lead);  // this warp is done with the query slot
                    return true;
                };
                if (N > 0) ok = issue_scores(0);
                for (int n = 0; n < N && ok; ++n) {
                    const int i = n / G, r = n - i * G, s = i % NKV1, yb = n % NY;
                    const int tb = n % NAT;
                    const bool look = n + 1 < N && (r + 1 < G || NKV1 >= 2);
                    if (look) {
                        ok = issue_scores(n + 1);
                        if (!ok) break;
                    }
                    ok = warp_wait(&at_full[tb], (n / NAT) & 1, err, kErrATFull);
                    if (!ok) break;
                    // the read-out of item n (warp 14) starts this Y^T buffer: complete first
                    ok = warp_wait(&inter_cmp[yb], (n / NY) & 1, err, kErrStateDone);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t tY = tmem + Cf::kColY + 64 * yb;
                    const uint64_t dv0 = sdesc_sw128(smem_u32(Vb(s)), 8192, 1024);
                    const uint64_t dh0 = sdesc_sw128(smem_u32(ATh(tb)), 16, 1024);
                    const uint64_t dl0 = sdesc_sw128(smem_u32(ATl(tb)), 16, 1024);
#pragma unroll 1
                    for (int ks = 0; ks < kC / 16; ++ks) {
                        const uint64_t av = dv0 + (uint64_t)(ks * 2048 >> 4);
                        mma_ss(tY, av, dh0 + (uint64_t)(ks * 32 >> 4), id_intra, 1, lead);
                        if (ALO) mma_ss(tY, av, dl0 + (uint64_t)(ks * 32 >> 4), id_intra, 1, lead);
                    }
                    mma_commit(&y_full[yb], lead);
                    if (r == G - 1) mma_commit(&empty_kv[s], lead);  // this warp is done with the K/V slot
                    if (!look && n + 1 < N) ok = issue_scores(n + 1);
                }
                } else {
                // scores and intra products; the read-outs and updates are warp 14's
                const int N = nck * G;
                for (int n = 0; n < N && ok; ++n) {
                    const int i = n / G, r = n - i * G, s = i % NKV1, sq = n % NQ1, ab = n % NA, yb = n % NY;
                    const int tb = n % NAT;
                    if (r == 0) {
                        ok = warp_wait(&conv_kv[s], (i / NKV1) & 1, err, kErrConvKV);
                        if (!ok) break;
                        tc_fence_after();
                    }
                    ok = warp_wait(&conv_q[sq], (n / NQ1) & 1, err, kErrConvQ);
                    if (!ok) break;
                    tc_fence_after();
                    if (n >= NA) {
                        ok = warp_wait(&a_empty[ab], ((n / NA) & 1) ^ 1, err, kErrAEmpty);
                        if (!ok) break;
                        tc_fence_after();
                    }
                    // scores, and in columns 64..71 phi(q).[Z_hi; Z_lo] from the Z rows
                    const uint32_t tA = tmem + Cf::kColA + 80 * ab;
                    const uint64_t dq0 = sdesc_sw128(smem_u32(Qb(sq)), 16, 1024);
                    const uint64_t dk0 = sdesc_sw128(smem_u32(Kb(s)), 16, 1024);
#pragma unroll 1
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint32_t qo = (ks >> 2) * 8192 + (ks & 3) * 32;
                        const uint32_t ko = (ks >> 2) * Cf::kKBlk + (ks & 3) * 32;
                        mma_ss(tA, dq0 + (qo >> 4), dk0 + (ko >> 4), id_scores, ks > 0, lead);
                    }
                    mma_commit(&a_full[ab], lead);
                    mma_commit(&empty_q[sq], lead);  // this warp is done with the query slot
                    ok = warp_wait(&at_full[tb], (n / NAT) & 1, err, kErrATFull);
                    if (!ok) break;
                    // the read-out of item n (warp 14) starts this Y^T buffer: complete first
                    ok = warp_wait(&inter_cmp[yb], (n / NY) & 1, err, kErrStateDone);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t tY = tmem + Cf::kColY + 64 * yb;
                    const uint64_t dv0 = sdesc_sw128(smem_u32(Vb(s)), 8192, 1024);
                    const uint64_t dh0 = sdesc_sw128(smem_u32(ATh(tb)), 16, 1024);
                    const uint64_t dl0 = sdesc_sw128(smem_u32(ATl(tb)), 16, 1024);
#pragma unroll 1
                    for (int ks = 0; ks < kC / 16; ++ks) {
                        const uint64_t av = dv0 + (uint64_t)(ks * 2048 >> 4);
                        mma_ss(tY, av, dh0 + (uint64_t)(ks * 32 >> 4), id_intra, 1, lead);
                        if (ALO) mma_ss(tY, av, dl0 + (uint64_t)(ks * 32 >> 4), id_intra, 1, lead);
                    }
                    mma_commit(&y_full[yb], lead);
                    if (r == G - 1) mma_commit(&empty_kv[s], lead);  // this warp is done with the K/V slot
                }
                }
                mma_commit(final_done, lead);  // every operation of this warp complete
            } else {
            for (int i = 0; i < nck && ok; ++i) {
                const int s = i % NKV1;
                if (Cf::kHasKV) {
                    ok = warp_wait(&conv_kv[s], (i / NKV1) & 1, err, kErrConvKV);
                    if (!ok) break;
                    tc_fence_after();
                }
                if (MODE == kState) {
                    if (GATED || i == 0) {
                        // the converters publish the (decayed) state before each update
                        ok = warp_wait(state_ready, i & 1, err, kErrStateReady);
                        if (!ok) break;
                        tc_fence_after();
                    }
                    issue_state_update(s);
                    // the non-gated state pass has no per-chunk hand-off: one phase at the end
                    if (GATED || i == nck - 1) mma_commit(state_done, lead);
                    mma_commit(&empty_kv[s], lead);
                    continue;
                }
                for (int r = 0; r < G && ok; ++r) {
                    const int n = i * G + r, sq = n % NQ1, ab = n % NA, yb = n % NY;
                    ok = warp_wait(&conv_q[sq], (n / NQ1) & 1, err, kErrConvQ);
                    if (!ok) break;
                    tc_fence_after();
                    // operand of the inter read-out: the queries (linear rule, gated exact
                    // chunk of one group) or the copy (decayed, or zero after a restart)
                    uint8_t* qop = (GATED && Gc(s)[kGFlag] != 1.f) ? Qd(sq) : Qb(sq);
                    const uint32_t tA = tmem + Cf::kColA + 80 * ab;
                    if (MODE == kCausal || NORM) {
                        if (n >= NA) {
                            ok = warp_wait(&a_empty[ab], ((n / NA) & 1) ^ 1, err, kErrAEmpty);
                            if (!ok) break;
                            tc_fence_after();
                        }
                        if (MODE == kCausal) {
                            // scores, and in columns 64..71 phi(q).[Z_hi; Z_lo] from the Z rows
                            const uint64_t dq0 = sdesc_sw128(smem_u32(Qb(sq)), 16, 1024);
                            const uint64_t dk0 = sdesc_sw128(smem_u32(Kb(s)), 16, 1024);
#pragma unroll kUnr
                            for (int ks = 0; ks < D / 16; ++ks) {
                                const uint32_t qo = (ks >> 2) * 8192 + (ks & 3) * 32;
                                const uint32_t ko = (ks >> 2) * Cf::kKBlk + (ks & 3) * 32;
                                mma_ss(tA, dq0 + (qo >> 4), dk0 + (ko >> 4), id_scores, ks > 0, lead);
                            }
                        } else {
#pragma unroll 1
                            for (int ks = 0; ks < D / 16; ++ks) {
                                const uint32_t qo = (ks >> 2) * 8192 + (ks & 3) * 32;
                                mma_ss(tA + 64, sdesc_sw128(smem_u32(Qb(sq) + qo), 16, 1024),
                                       sdesc_sw128(smem_u32(zr_at(0, ks >> 2) + (ks & 3) * 32), 16, 1024), id_qz,
                                       ks > 0, lead);
                            }
                        }
                        mma_commit(&a_full[ab], lead);
                    }
                    if (r == 0 && (MODE == kCausal || i == 0)) {
                        if (TF32 && MODE == kCausal && i > 0)  // the update of chunk i-1 has completed
                            ok = warp_wait(state_done, (i - 1) & 1, err, kErrStateDone);
                        else  // start state in place (tf32), or the hi/lo copy of S(i) (gated)
                            ok = warp_wait(state_ready, (MODE == kCausal && !TF32) ? (i & 1) : 0, err,
                                           kErrStateReady);
                        if (!ok) break;
                        tc_fence_after();
                    }
                    if (n >= NY) {
                        ok = warp_wait(&y_empty[yb], ((n / NY) & 1) ^ 1, err, kErrYEmpty);
                        if (!ok) break;
                        tc_fence_after();
                    }
                    // inter: Y^T = S_prev^T . Q^T (tf32 from the fp32 state, or hi + lo)
                    const uint32_t tY = tmem + Cf::kColY + 64 * yb;
                    if (TF32) {
                        const uint64_t df0 = sdesc_sw128(smem_u32(Qf(sq)), 16, 1024);
#pragma unroll kUnr
                        for (int ks = 0; ks < D / 8; ++ks) {
                            const uint32_t ko = (ks >> 2) * 8192 + (ks & 3) * 32;
                            mma_ts_tf32(tY, tS + ks * 8, df0 + (ko >> 4), id_inter_tf32, ks > 0, lead);
                        }
                    } else {
#pragma unroll 1
                        for (int ks = 0; ks < D / 16; ++ks) {
                            const uint32_t ko = (ks >> 2) * 8192 + (ks & 3) * 32;
                            const uint64_t bq = sdesc_sw128(smem_u32(qop + ko), 16, 1024);
                            mma_ts(tY, tHi + ks * 8, bq, id_inter, ks > 0, lead);
                            mma_ts(tY, tLo + ks * 8, bq, id_inter, 1, lead);
                        }
                    }
                    mma_commit(&empty_q[sq], lead);
                    if (MODE == kCausal) {
                        if (!TF32 && r == G - 1) {
                            // every read-out of this chunk is issued (from the hi/lo
                            // copy): update the state now
                            issue_state_update(s);
                            mma_commit(state_done, lead);
                        }
                        if (TF32 && r == G - 1) mma_commit(inter_done, lead);
                        const int tb = n % NAT;
                        ok = warp_wait(&at_full[tb], (n / NAT) & 1, err, kErrATFull);
                        if (!ok) break;
                        tc_fence_after();
                        // intra: Y^T += V^T . A^T (hi [+ lo])
                        const uint64_t dv0 = sdesc_sw128(smem_u32(Vb(s)), 8192, 1024);
                        const uint64_t dh0 = sdesc_sw128(smem_u32(ATh(tb)), 16, 1024);
                        const uint64_t dl0 = sdesc_sw128(smem_u32(ATl(tb)), 16, 1024);
#pragma unroll kUnr
                        for (int ks = 0; ks < kC / 16; ++ks) {
                            const uint64_t av = dv0 + (uint64_t)(ks * 2048 >> 4);
                            mma_ss(tY, av, dh0 + (uint64_t)(ks * 32 >> 4), id_intra, 1, lead);
                            if (ALO) mma_ss(tY, av, dl0 + (uint64_t)(ks * 32 >> 4), id_intra, 1, lead);
                        }
                    }
                    mma_commit(&y_full[yb], lead);
                    if (TF32 && MODE == kCausal && r == G - 1) {
                        // the update overwrites the state that this chunk's read-outs
                        // take as their A operand: only after they have completed
                        ok = warp_wait(inter_done, i & 1, err, kErrStateDone);
                        if (!ok) break;
                        tc_fence_after();
                        issue_state_update(s);
                        mma_commit(state_done, lead);
                    }
                }
                if (!ok) break;
                if (Cf::kHasKV) mma_commit(&empty_kv[s], lead);
            }
            // last: every operation above has completed (also after an early exit)
            if (TF32 && MODE == kCausal) mma_commit(final_done, lead);
            }
        }
    } else if (warp < kEpiWarp0) {
        // -------------------------------------------------------- state warps
        // Own the carried state in TMEM: the start state, its bf16 hi/lo copy
        // for each chunk's read-out (the only loop-carried hand-off), the
        // per-chunk decay of the gated rule, and the final state.
        const int quad = warp & 3;  // TMEM lane quadrant of this warp
        const int st_t = tid - kStateWarp0 * 32;
        const bool m64 = D == 64;
        const int vrow = m64 ? (quad * 16 + lane) : (quad * 32 + lane);  // value row of S^T in this lane
        const bool vrow_ok = m64 ? lane < 16 : true;
        bool ok = true;

        // ---- start state -> S^T (fp32) in TMEM.  Causal segment s > 0 folds
        // the increments of segments 0..s-1 (from the state pass, fold_r per
        // segment) onto the initial state, decay-weighted for gated.
        const bool fold = MODE == kCausal && a.S_seg && seg > 0;
        const int nfold = seg * a.fold_r, fstride = nseg * a.fold_r;  // increments to fold; per (b, kv head)
        const float* S_start = MODE == kState ? nullptr : a.S_init;
        if (MODE == kCausal) griddep_wait();  // the segment state pass has completed
        // Loads are batched 32 columns x 2 segments at a time (independent
        // addresses, all in flight together); the additions keep the segment
        // order 0, 1, ..., seg-1.
        for (int c0 = 0; c0 < D; c0 += 32) {
            float run[32];
#pragma unroll
            for (int x = 0; x < 32; ++x)
                run[x] = (S_start && vrow_ok) ? S_start[(size_t)bh * D * D + (size_t)(c0 + x) * D + vrow] : 0.f;
            if (fold && vrow_ok) {
                for (int p = 0; p < nfold; p += 2) {
                    const bool two = p + 1 < nfold;
                    const float* s0 = a.S_seg + ((size_t)bh * fstride + p) * D * D + (size_t)c0 * D + vrow;
                    const float* s1 = s0 + (size_t)D * D;
                    float d0[32], d1[32];
#pragma unroll
                    for (int x = 0; x < 32; ++x) {
                        d0[x] = s0[(size_t)x * D];
                        d1[x] = two ? s1[(size_t)x * D] : 0.f;
                    }
                    const float w0 = GATED ? __expf(a.G_seg[(size_t)bh * fstride + p]) : 1.f;
                    const float w1 = (GATED && two) ? __expf(a.G_seg[(size_t)bh * fstride + p + 1]) : 1.f;
#pragma unroll
                    for (int x = 0; x < 32; ++x) {
                        run[x] = GATED ? fmaf(w0, run[x], d0[x]) : run[x] + d0[x];
                        if (two) run[x] = GATED ? fmaf(w1, run[x], d1[x]) : run[x] + d1[x];
                    }
                }
            }
            uint32_t r[32];
#pragma unroll
            for (int x = 0; x < 32; ++x) r[x] = __float_as_uint(run[x]);
            tmem_st32(tmem_addr(tmem + Cf::kColS, quad * 32, c0), r);
        }
        tmem_st_wait();
        float gsum = 0.f;  // gated, state mode: total log decay of the segment

        // ---- state hi/lo (and, gated, the decay of the fp32 state in place)
        // hi/lo copy of hl_mul * S for the read-out; S <- decay_mul * S in place
        auto convert_state = [&](float decay_mul, bool write_back, float hl_mul = 1.f) {
#pragma unroll 1
            for (int c0 = 0; c0 < D; c0 += 64) {
                uint32_t r0[32], r1[32];
                tmem_ld32(tmem_addr(tmem + Cf::kColS, quad * 32, c0), r0);
                tmem_ld32(tmem_addr(tmem + Cf::kColS, quad * 32, c0 + 32), r1);
                tmem_ld_wait();
                reg_fence(r0);
                reg_fence(r1);
                if (MODE != kState) {
                    uint32_t h0[16], l0[16], h1[16], l1[16];
#pragma unroll
                    for (int x = 0; x < 16; ++x) {
                        split2(hl_mul * __uint_as_float(r0[2 * x]), hl_mul * __uint_as_float(r0[2 * x + 1]), h0[x], l0[x]);
                        split2(hl_mul * __uint_as_float(r1[2 * x]), hl_mul * __uint_as_float(r1[2 * x + 1]), h1[x], l1[x]);
                    }
                    tmem_st16(tmem_addr(tmem + Cf::kColHi, quad * 32, c0 / 2), h0);
                    tmem_st16(tmem_addr(tmem + Cf::kColHi, quad * 32, c0 / 2 + 16), h1);
                    tmem_st16(tmem_addr(tmem + Cf::kColLo, quad * 32, c0 / 2), l0);
                    tmem_st16(tmem_addr(tmem + Cf::kColLo, quad * 32, c0 / 2 + 16), l1);
                }
                if (write_back) {
#pragma unroll
                    for (int x = 0; x < 32; ++x) {
                        r0[x] = __float_as_uint(__uint_as_float(r0[x]) * decay_mul);
                        r1[x] = __float_as_uint(__uint_as_float(r1[x]) * decay_mul);
                    }
                    tmem_st32(tmem_addr(tmem + Cf::kColS, quad * 32, c0), r0);
                    tmem_st32(tmem_addr(tmem + Cf::kColS, quad * 32, c0 + 32), r1);
                }
            }
            tmem_st_wait();
        };
        auto publish_state = [&]() {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(state_ready);
        };

        if (MODE == kApply) {
            // fixed global state (hi/lo once for the gated layout)
            tc_fence_after();
            if (!TF32) convert_state(1.f, false);
            publish_state();
        } else if ((MODE == kState && !GATED) || (MODE == kCausal && TF32)) {
            // the start (or zero) state is in place; the tensor core reads and
            // updates it without further hand-offs
            publish_state();
        } else {
            // Gated causal: these warps also run the output stage, between the
            // state conversions.  Per chunk i: outputs of heads 0..G-3 of chunk
            // i-1, the conversion of S(i), then heads G-2 and G-1 of chunk i-1.
            // The update of chunk i-1 (which S(i) waits for) follows the read-out
            // of its last head, which needs the Y buffer of head G-3 released
            // first, so those outputs must come before the conversion.
            constexpr bool kOut = MODE == kCausal;
            // output row factors of exact chunks (two per lane), for the chunk
            // being converted (cur) and the one before it (prev), whose outputs
            // are emitted around this conversion
            float eo_cur_lo = 1.f, eo_cur_hi = 1.f, eo_prev_lo = 1.f, eo_prev_hi = 1.f;
            bool ex_cur = false, ex_prev = false;
            for (int i = 0; i < nck && ok; ++i) {
                // (cur still holds chunk i - 1 here)
                if (kOut && i > 0)
                    for (int r = 0; r < G - 2 && ok; ++r) ok = emit_y((i - 1) * G + r, eo_cur_lo, eo_cur_hi, ex_cur);
                if (!ok) break;
                // S(i): after the update of chunk i-1 and every read-out that used S_prev
                if (i > 0) {
                    ok = warp_wait(state_done, (i - 1) & 1, err, kErrStateDone);
                    if (!ok) break;
                }
                float gtot = 0.f, hl_mul = 1.f;
                if (GATED) {
                    // the decay of chunk i comes with its converted keys
                    const int s = i % NKV1;
                    ok = warp_wait(&conv_kv[s], (i / NKV1) & 1, err, kErrConvKV);
                    if (!ok) break;
                    const float* gc = Gc(s);
                    gtot = gc[kGTot];
                    eo_prev_lo = eo_cur_lo, eo_prev_hi = eo_cur_hi, ex_prev = ex_cur;
                    ex_cur = gc[kGFlag] != 0.f;
                    eo_cur_lo = ex_cur ? gc[lane] : 1.f;
                    eo_cur_hi = ex_cur ? gc[lane + 32] : 1.f;
                    if (ex_cur) hl_mul = __expf(gc[kGRef]);
                }
                tc_fence_after();
                convert_state(GATED ? __expf(gtot) : 1.f, GATED, hl_mul);
                publish_state();
                if (MODE == kState) gsum += gtot;
                if (kOut && i > 0)
                    for (int r = max(0, G - 2); r < G && ok; ++r)
                        ok = emit_y((i - 1) * G + r, eo_prev_lo, eo_prev_hi, ex_prev);
            }
            if (kOut && nck > 0)
                for (int r = 0; r < G && ok; ++r) ok = emit_y((nck - 1) * G + r, eo_cur_lo, eo_cur_hi, ex_cur);
        }
        if (TF32 && MODE != kState) {
            // linear rule: the state needs no per-chunk work here, so these
            // warps run the output stage, beside the score warps
            for (int m = 0; m < nck * G && ok; ++m) ok = emit_y(m);
        }

        // ---- final state out: causal (last segment) or every segment in state mode
        const bool write_state =
            ok && nck > 0 && ((MODE == kCausal && seg == nseg - 1 && a.S_dst) || MODE == kState);
        if (MODE == kCausal && TF32 && nck > 0) {
            // the last update is not followed by any read-out: wait for it here,
            // also when no state is written, before TMEM is released
            ok = warp_wait(final_done, 0, err, kErrStateDone) && ok;
            tc_fence_after();
        }
        if (write_state && ok) {
            // gated causal: phase nck-1 (one per chunk); non-gated state pass: its single phase
            if (!(MODE == kCausal && TF32))
                ok = warp_wait(state_done, (MODE == kState && !GATED) ? 0 : ((nck - 1) & 1), err, kErrStateDone);
            tc_fence_after();
            if (ok) {
                float* Sd = MODE == kState ? a.S_dst + ((size_t)bh * nseg + seg) * D * D : a.S_dst + (size_t)bh * D * D;
#pragma unroll 1
                for (int c0 = 0; c0 < D; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld32(tmem_addr(tmem + Cf::kColS, quad * 32, c0), r);
                    tmem_ld_wait();
                    reg_fence(r);
                    if (vrow_ok)
#pragma unroll
                        for (int x = 0; x < 32; ++x) Sd[(size_t)(c0 + x) * D + vrow] = __uint_as_float(r[x]);
                }
                if (MODE == kState && GATED && st_t == 0) a.G_dst[(size_t)bh * nseg + seg] = gsum;
            }
        }
    } else if (warp < Cf::kFeatW0) {
        // -------------------------------------------------------------- epilogue
        const int quad = warp & 3;  // TMEM lane quadrant of this warp
        const int n_total = Cf::kHasQ ? nck * G : 0;
        const int et = tid - kEpiWarp0 * 32;  // 0..127
        bool ok = true;
        if (kQOnEpi && n_total > 0) ok = q_features(0, 0, et);
        for (int n = 0; n < n_total && ok; ++n) {
            {
                // -------- scores of item n: mask, decay, hi/lo split, 1/den
                const int ab = n % NA;
                const int s = (n / G) % NKV1;
                if (MODE == kCausal || NORM) {
                    ok = warp_wait(&a_full[ab], (n / NA) & 1, err, kErrAFull);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t tA = tmem + Cf::kColA + 80 * ab;
                    // The 64 x 64 score tile (M = 64: TMEM lanes 0-15 of each quadrant)
                    // read in the 16x256b shape, so that all 32 lanes work: this
                    // thread holds rows r1 = 16 quad + lane/4 and r2 = r1 + 8, columns
                    // 8g + cq and 8g + cq + 1 of each 8-column group g.  One round
                    // trip to TMEM; the buffer is released before the masking.
                    const int r1 = quad * 16 + (lane >> 2), r2 = r1 + 8, cq = 2 * (lane & 3);
                    const uint32_t tq = tmem_addr(tA, quad * 32, 0);
                    uint32_t sc[32], zz[4];
                    if (MODE == kCausal) tmem_ld16x256b_x8(tq, sc);
                    if (NORM) tmem_ld16x256b_x1(tq + 64, zz);  // columns 64, 65: phi(q).[Z_hi, Z_lo]
                    tmem_ld_wait();
                    if (MODE == kCausal) reg_fence(sc);
                    if (NORM) reg_fence(zz);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&a_empty[ab]);  // TMEM scores read out
                    float den1 = 1.f, den2 = 1.f;
                    if (NORM) {
                        // phi(q).Z_prev sits in the thread of column pair 0 of each row
                        const int src = lane & ~3;
                        den1 = __shfl_sync(0xffffffffu, __uint_as_float(zz[0]) + __uint_as_float(zz[1]), src) + eps;
                        den2 = __shfl_sync(0xffffffffu, __uint_as_float(zz[2]) + __uint_as_float(zz[3]), src) + eps;
                    }
                    if (MODE == kCausal) {
                        const float* gc = reinterpret_cast<const float*>(Gc(s));
                        const int tb = n % NAT;
                        if (n >= NAT) {
                            // the intra product that read this buffer last (item n - NAT)
                            // has completed: its completion is the y_full phase of that item
                            ok = warp_wait(&y_full[(n - NAT) % NY], ((n - NAT) / NY) & 1, err, kErrATEmpty);
                            if (!ok) break;
                            tc_fence_after();
                        }
                        // masked rows (decay-weighted for the gated rule: w1(j), w2(j)
                        // are exp(G_i - G_j) for rows r1, r2), bf16 hi [+ lo] pairs into
                        // the swizzled A^T tile, and the row sums for the normalizer
                        auto mask_rows = [&](auto w1, auto w2) {
                            float p1 = 0.f, p2 = 0.f;
#pragma unroll
                            for (int g = 0; g < 8; ++g) {
                                const int j = 8 * g + cq;
                                float a0 = j <= r1 ? __uint_as_float(sc[4 * g]) : 0.f;
                                float a1 = j + 1 <= r1 ? __uint_as_float(sc[4 * g + 1]) : 0.f;
                                float b0 = j <= r2 ? __uint_as_float(sc[4 * g + 2]) : 0.f;
                                float b1 = j + 1 <= r2 ? __uint_as_float(sc[4 * g + 3]) : 0.f;
                                if (NORM) {
                                    p1 += a0 + a1;
                                    p2 += b0 + b1;
                                }
                                if (GATED) {
                                    if (j <= r1) a0 *= w1(j);
                                    if (j + 1 <= r1) a1 *= w1(j + 1);
                                    if (j <= r2) b0 *= w2(j);
                                    if (j + 1 <= r2) b1 *= w2(j + 1);
                                }
                                const uint32_t o1 = (uint32_t)(r1 * 128 + ((g ^ (r1 & 7)) << 4) + 2 * cq);
                                const uint32_t o2 = (uint32_t)(r2 * 128 + ((g ^ (r2 & 7)) << 4) + 2 * cq);
                                if (ALO) {
                                    uint32_t h1, l1, h2, l2;
                                    split2(a0, a1, h1, l1);
                                    split2(b0, b1, h2, l2);
                                    *reinterpret_cast<uint32_t*>(ATh(tb) + o1) = h1;
                                    *reinterpret_cast<uint32_t*>(ATl(tb) + o1) = l1;
                                    *reinterpret_cast<uint32_t*>(ATh(tb) + o2) = h2;
                                    *reinterpret_cast<uint32_t*>(ATl(tb) + o2) = l2;
                                } else {
                                    *reinterpret_cast<uint32_t*>(ATh(tb) + o1) = bf2_bits(__floats2bfloat162_rn(a0, a1));
                                    *reinterpret_cast<uint32_t*>(ATh(tb) + o2) = bf2_bits(__floats2bfloat162_rn(b0, b1));
                                }
                            }
                            if (NORM) {  // row sums over the four threads of a row
                                p1 += __shfl_xor_sync(0xffffffffu, p1, 1);
                                p1 += __shfl_xor_sync(0xffffffffu, p1, 2);
                                p2 += __shfl_xor_sync(0xffffffffu, p2, 1);
                                p2 += __shfl_xor_sync(0xffffffffu, p2, 2);
                                den1 += p1;
                                den2 += p2;
                            }
                        };
                        if constexpr (GATED) {
                            if (gc[kGFlag] == 1.f) {
                                // exact chunk: exp(G_i - G_j) = exp(G_i - ref) * exp(ref - G_j);
                                // the row factor is applied to the output row, so the
                                // weights are the column factors of the feature warps
                                const float* ef = gc + kGCol;
                                mask_rows([&](int j) { return ef[j]; }, [&](int j) { return ef[j]; });
                            } else if (gc[kGFlag] == 2.f) {
                                // exact chunk with restarts: zero across groups
                                const float* ef = gc + kGCol;
                                const uint64_t word = gc_word(gc);
                                mask_rows([&](int j) { return same_group(word, j, r1) ? ef[j] : 0.f; },
                                          [&](int j) { return same_group(word, j, r2) ? ef[j] : 0.f; });
                            } else {
                                const float g1 = gc[r1], g2 = gc[r2];
                                mask_rows([&](int j) { return __expf(g1 - gc[j]); },
                                          [&](int j) { return __expf(g2 - gc[j]); });
                            }
                        } else {
                            mask_rows([](int) { return 1.f; }, [](int) { return 1.f; });
                        }
                    }
                    if (MODE == kCausal) {
                        fence_proxy_async();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&at_full[n % NAT]);
                    }
                    if (NORM) {
                        // hand scale/den to the output stage (without the normalizer
                        // the factor is the constant scale and needs no hand-off)
                        if ((lane & 3) == 0) {
                            inv_den[(n & 3) * 64 + r1] = scale / den1;
                            inv_den[(n & 3) * 64 + r2] = scale / den2;
                        }
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&den_full[n & 3]);
                    }
                }
            }
            // the next query item, while the tensor core runs this item's products
            if (kQOnEpi && ok && n + 1 < n_total) ok = q_features((n + 1) / G, n + 1, et);
        }
    } else if (warp == kIdleWarp) {
        // ------------------------------------------------ MMA issuer of the state
        // (split issue only): per chunk, the read-out of every query head with
        // the carried fp32 state (kind::tf32, state from TMEM as A), then the
        // state update once those read-outs have completed.
        if constexpr (split) {
            const uint32_t lead = lane == 0;
            bool ok = true;
            constexpr uint32_t id_inter_tf32 = idesc_tf32(D, 64);
            constexpr uint32_t id_state = idesc_bf16(D, D, true, true);
            const uint32_t tS = tmem + Cf::kColS;
            constexpr int kUnr2 = 1;
            for (int i = 0; i < nck && ok; ++i) {
                const int s = i % NKV1;
                // S before chunk i: the start state (state warps) or this warp's last update
                ok = i == 0 ? warp_wait(state_ready, 0, err, kErrStateReady)
                            : warp_wait(upd_done, (i - 1) & 1, err, kErrStateDone);
                if (!ok) break;
                tc_fence_after();
                int n = i * G;
                for (int r = 0; r < G && ok; ++r) {
                    n = i * G + r;
                    const int sq = n % NQ1, yb = n % NY;
                    ok = warp_wait(&conv_q[sq], (n / NQ1) & 1, err, kErrConvQ);
                    if (!ok) break;
                    if (n >= NY) ok = warp_wait(&y_empty[yb], ((n / NY) & 1) ^ 1, err, kErrYEmpty);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t tY = tmem + Cf::kColY + 64 * yb;
                    const uint64_t df0 = sdesc_sw128(smem_u32(Qf(sq)), 16, 1024);
#pragma unroll kUnr2
                    for (int ks = 0; ks < D / 8; ++ks) {
                        const uint32_t ko = (ks >> 2) * 8192 + (ks & 3) * 32;
                        mma_ts_tf32(tY, tS + ks * 8, df0 + (ko >> 4), id_inter_tf32, ks > 0, lead);
                    }
                    mma_commit(&empty_q[sq], lead);     // this warp is done with the query slot
                    mma_commit(&inter_cmp[yb], lead);   // the intra product may add to Y^T
                }
                if (!ok) break;
                // the update overwrites S, which the read-outs take as their A
                // operand: wait for the last one (and with it every earlier one)
                ok = warp_wait(&inter_cmp[n % NY], (n / NY) & 1, err, kErrStateDone);
                if (!ok) break;
                ok = warp_wait(&conv_kv[s], (i / NKV1) & 1, err, kErrConvKV);
                if (!ok) break;
                tc_fence_after();
                // S^T += V^T . phi(K) (+ V^T . phi(K)_lo)
                const uint64_t dv0 = sdesc_sw128(smem_u32(Vb(s)), 8192, 1024);
                const uint64_t dk0 = sdesc_sw128(smem_u32(Kb(s)), (uint32_t)Cf::kKBlk, 1024);
                const uint64_t dl0 = sdesc_sw128(smem_u32(Klo(s)), 8192, 1024);
#pragma unroll kUnr2
                for (int ks = 0; ks < kC / 16; ++ks) {
                    const uint64_t o = (uint64_t)(ks * 2048 >> 4);
                    mma_ss(tS, dv0 + o, dk0 + o, id_state, 1, lead);
                    if (SPLITK) mma_ss(tS, dv0 + o, dl0 + o, id_state, 1, lead);
                }
                mma_commit(&empty_kv[s], lead);  // this warp is done with the K/V slot
                mma_commit(upd_done, lead);
            }
            mma_commit(final_done, lead);  // every operation of this warp complete
        }
    } else if (!split || warp != 13) {
        // ------------------------------------------------------ feature warps
        // Feature maps of keys and queries in shared memory (bf16 hi, lo part
        // of the keys for the state update), decayed copies for the gated
        // rule, the Z rows of every chunk and the running key sum Z.  Runs
        // ahead of the state chain, limited only by the load rings.
        constexpr int kCPR = Cf::kCPR, kRowStep = Cf::kRowStep, kPer = Cf::kPer;
        const int fslot = kFeatMove && warp == kFeatMovedTo ? 13 - Cf::kFeatW0 : warp - Cf::kFeatW0;
        const int ct = fslot * 32 + lane;  // 0 .. kFeatThreads - 1
        const int cc = ct % kCPR;              // 16-byte chunk column: features 8cc..8cc+7
        const int rbase = ct / kCPR;           // rows rbase + kRowStep * m
        bool ok = true;
        uint32_t gphase = 0;
        int zbuf = 0;
        // 16-byte chunk m of this thread in a swizzled 64 x D tile whose
        // 64-feature blocks are `blk` bytes apart
        auto chunk_off = [&](int m, int blk = 8192) -> uint32_t {
            const int row = rbase + kRowStep * m;
            return static_cast<uint32_t>((cc >> 3) * blk + row * 128 + ((((cc & 7) ^ (row & 7))) << 4));
        };
        // element (Z row r, feature k) of the Z rows of stage s
        auto zr_elem = [&](int s, int r, int k) -> __nv_bfloat16& {
            return bf_at(zr_at(s, k >> 6), sw128_offset(r, (k & 63) * 2));
        };

        // zero the constant rows 2..7 of every Z-row block
        if (NORM && MODE != kState) {
            const int nzr = MODE == kApply ? 1 : NKV;
            for (int z = 0; z < nzr; ++z)
                for (int e = ct; e < D * 6; e += Cf::kFeatThreads) zr_elem(z, 2 + e / D, e % D) = __float2bfloat16(0.f);
        }
        // running key sum Z in a register of thread k < D (state pass: the increment)
        float zreg = 0.f;
        // start key sum: the initial Z plus, for a later sequence segment, the
        // increments of the earlier ones (written by the segment state pass:
        // its completion is awaited first)
        auto start_z = [&]() {
            griddep_wait();
            const bool fold = MODE == kCausal && a.S_seg && seg > 0;
            zreg = a.Z_init ? a.Z_init[(size_t)bh * D + ct] : 0.f;
            if (fold && a.Z_seg) {
                // independent loads, four in flight; summed in segment order
                const int nfold = seg * a.fold_r, fstride = nseg * a.fold_r;
                for (int p = 0; p < nfold; p += 4) {
                    float z4[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        z4[u] = p + u < nfold ? a.Z_seg[((size_t)bh * fstride + p + u) * D + ct] : 0.f;
#pragma unroll
                    for (int u = 0; u < 4; ++u) zreg += z4[u];
                }
            }
        };
        if (NORM && ct < D && MODE == kApply) start_z();

        // ---- keys of chunk i: feature map (+ lo part), decayed keys, Z rows and sums
        // mask bytes of the next chunk, loaded one chunk ahead (their latency
        // hides behind the wait for that chunk's tiles)
        uint32_t mb_next = mask_bytes(c_begin * kC);
        auto process_kv = [&](int i) -> bool {
            const int s = i % NKV1;
            const int t0 = (c_begin + i) * kC;
            const int valid = min(kC, T - t0);
            const uint32_t mb = mb_next;
            if (mask && i + 1 < nck) mb_next = mask_bytes(t0 + kC);
            if (!warp_wait(&full_kv[s], (i / NKV1) & 1, err, kErrFullKV)) return false;
            // invalid steps (mask): their phi(k) and v rows become zero, so
            // they add nothing to the state, the key sum or any score
            const uint64_t okw = valid_bits(mb);
            float* gc = Gc(s);
            float gtot = 0.f;
            bool gx = false;     // exact chunk (kGFlag)
            float e_tr = 0.f;    // exact chunk: exp(gtot - ref of the last group)
            uint64_t gword = 0;  // exact chunk: restart steps
            if (GATED) {
                // inclusive cumulative log decay inside the chunk (first converter warp)
                if (ct < 32) {
                    float g0 = 0.f, g1 = 0.f;
                    const int j0 = 2 * ct, j1 = 2 * ct + 1;
                    // an invalid step (mask) keeps the state: no decay either
                    // a log decay of -inf (or any value below kMinLogDecay) is
                    // taken as kMinLogDecay: exp of it, and of every cumulative
                    // difference that crosses it, is zero in float32 -- the same
                    // "forget everything" restart -- while the differences of the
                    // later steps of the chunk stay finite (no -inf - -inf)
                    if (j0 < valid && ((okw >> j0) & 1))
                        g0 = fmaxf(__bfloat162float(decay[((size_t)b * T + t0 + j0) * Hkv + hk]), kMinLogDecay);
                    if (j1 < valid && ((okw >> j1) & 1))
                        g1 = fmaxf(__bfloat162float(decay[((size_t)b * T + t0 + j1) * Hkv + hk]), kMinLogDecay);
                    const float sum = g0 + g1;
                    float incl = sum;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const float t = __shfl_up_sync(0xffffffffu, incl, o);
                        if (lane >= o) incl += t;
                    }
                    const float c0 = incl - sum + g0, c1 = incl;
                    // groups split at restart steps; a reference in the middle of each
                    // group's range; an exact chunk (every factor exp(+-(G - ref_g))
                    // within e^30, every ref below 30) keeps the factors instead of G
                    // (see kGCol)
                    const uint64_t word = restart_word(g0 <= kRestartLogDecay, g1 <= kRestartLogDecay);
                    const int ngroups = __popcll(word) + 1;
                    const uint64_t m0 = (2ull << j0) - 1, m1 = j1 == 63 ? ~0ull : (2ull << j1) - 1;
                    const int grp0 = __popcll(word & m0), grp1 = __popcll(word & m1);
                    bool exact = true;
                    float ref0 = 0.f, ref1 = 0.f, ref_first = 0.f, ref_last = 0.f;
#pragma unroll 1
                    for (int g = 0; g < ngroups; ++g) {
                        float mx = fmaxf(grp0 == g ? c0 : -INFINITY, grp1 == g ? c1 : -INFINITY);
                        float mn = fminf(grp0 == g ? c0 : INFINITY, grp1 == g ? c1 : INFINITY);
#pragma unroll
                        for (int o = 16; o > 0; o >>= 1) {
                            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                            mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
                        }
                        if (mx < mn) continue;  // empty group (a restart on step 0)
                        exact = exact && (mx - mn) < 60.f && mx < 30.f;
                        const float ref = 0.5f * (mx + mn);
                        if (grp0 == g) ref0 = ref;
                        if (grp1 == g) ref1 = ref;
                        if (g == 0) ref_first = ref;
                        ref_last = ref;
                    }
                    gc[j0] = exact ? __expf(c0 - ref0) : c0;
                    gc[j1] = exact ? __expf(c1 - ref1) : c1;
                    gc[kGCol + j0] = exact ? __expf(ref0 - c0) : 0.f;
                    gc[kGCol + j1] = exact ? __expf(ref1 - c1) : 0.f;
                    if (ct == 0) {
                        gc[kGRef] = ref_first;
                        gc[kGRefLast] = ref_last;
                        gc[kGFlag] = exact ? (ngroups > 1 ? 2.f : 1.f) : 0.f;
                        gc[kGWord0] = __uint_as_float((uint32_t)word);
                        gc[kGWord1] = __uint_as_float((uint32_t)(word >> 32));
                    }
                    if (ct == 31) gc[kGTot] = c1;  // G of the chunk's last step
                }
                if (!group_sync(conv_group, gphase, err, kErrStateReady)) return false;
                gtot = gc[kGTot];
                gx = gc[kGFlag] != 0.f;
                if (gx) {
                    e_tr = __expf(gtot - gc[kGRefLast]);
                    gword = gc_word(gc);
                }
            }
            const bool touch = GATED || SPLITK || NORM || fmap != LA_FMAP_NONE || mask;
            if (touch) {
                float colsum[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
                // A rolled loop: its body stays in the instruction cache across
                // iterations (the roles of this kernel share each sub-partition's
                // instruction cache, so straight-line code would be fetched anew
                // every chunk).
                // kDrop: the chunk holds invalid steps (mask), dropped row by row;
                // a chunk whose steps are all valid runs the unmasked loop
                auto conv_rows = [&](auto drop_tag) {
                constexpr bool kDrop = decltype(drop_tag)::value;
                uint4 nxt = *reinterpret_cast<const uint4*>(Kb(s) + chunk_off(0, Cf::kKBlk));
#pragma unroll 1
                for (int m = 0; m < kPer; ++m) {
                    const int row = rbase + kRowStep * m;
                    const uint4 cur = nxt;
                    if (m + 1 < kPer) nxt = *reinterpret_cast<const uint4*>(Kb(s) + chunk_off(m + 1, Cf::kKBlk));
                    const bool drop = kDrop && !((okw >> row) & 1);
                    if (drop) {
                        *reinterpret_cast<uint4*>(Kb(s) + chunk_off(m, Cf::kKBlk)) = make_uint4(0, 0, 0, 0);
                        *reinterpret_cast<uint4*>(Vb(s) + chunk_off(m)) = make_uint4(0, 0, 0, 0);
                    }
                    float f[8];
                    bf8_to_f(cur, f);
                    uint4 hi, lo;
                    if (GATED) {
                        // exp(G_C - G_row): from the column factor in an exact chunk
                        // (zero for steps before the chunk's last restart)
                        const float w = gx ? (same_group(gword, row, kC - 1) ? e_tr * gc[kGCol + row] : 0.f)
                                           : __expf(gtot - gc[row]);
#pragma unroll
                        for (int e = 0; e < 8; ++e) f[e] = drop ? 0.f : f[e] * w;
                        split8(f, hi, lo);
                        *reinterpret_cast<uint4*>(Kd(s) + chunk_off(m)) = hi;
                        *reinterpret_cast<uint4*>(Klo(s) + chunk_off(m)) = lo;
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) f[e] = drop ? 0.f : phi<true>(fmap, f[e], eps);
                        if (fmap != LA_FMAP_NONE || SPLITK) {
                            split8(f, hi, lo);
                            if (fmap != LA_FMAP_NONE) *reinterpret_cast<uint4*>(Kb(s) + chunk_off(m, Cf::kKBlk)) = hi;
                            if (SPLITK) *reinterpret_cast<uint4*>(Klo(s) + chunk_off(m)) = lo;
                        }
                        if (NORM && row < valid)
#pragma unroll
                            for (int e = 0; e < 8; ++e) colsum[e] += f[e];
                    }
                }
                };
                if (!mask || okw == ~0ull) {
                    conv_rows(BoolTag<false>{});
                } else if (okw == 0ull) {
                    // every step of the chunk invalid: zero key and value rows only
#pragma unroll 1
                    for (int m = 0; m < kPer; ++m) {
                        const uint4 z = make_uint4(0, 0, 0, 0);
                        *reinterpret_cast<uint4*>(Kb(s) + chunk_off(m, Cf::kKBlk)) = z;
                        *reinterpret_cast<uint4*>(Vb(s) + chunk_off(m)) = z;
                        if (GATED) *reinterpret_cast<uint4*>(Kd(s) + chunk_off(m)) = z;
                        if (SPLITK) *reinterpret_cast<uint4*>(Klo(s) + chunk_off(m)) = z;
                    }
                } else {
                    conv_rows(BoolTag<true>{});
                }
                if (NORM) {
                    // partial column sums of this chunk, reduced after the tile is released
                    float* zp = zpart + zbuf * Cf::kZpart;
                    *reinterpret_cast<float4*>(zp + rbase * D + 8 * cc) =
                        make_float4(colsum[0], colsum[1], colsum[2], colsum[3]);
                    *reinterpret_cast<float4*>(zp + rbase * D + 8 * cc + 4) =
                        make_float4(colsum[4], colsum[5], colsum[6], colsum[7]);
                    // Z rows of this chunk hold Z_prev (hi, lo): known before its sums
                    if (MODE != kState && ct < D) {
                        if (MODE == kCausal && i == 0) start_z();
                        const __nv_bfloat16 h = __float2bfloat16_rn(zreg);
                        zr_elem(s, 0, ct) = h;
                        zr_elem(s, 1, ct) = __float2bfloat16_rn(zreg - __bfloat162float(h));
                    }
                }
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(&conv_kv[s]);  // the tile goes to the tensor core
            if (touch && NORM) {
                // Z += this chunk's column sums, off the path to the tensor core
                const float* zp = zpart + zbuf * Cf::kZpart;
                if (!group_sync(conv_group, gphase, err, kErrStateReady)) return false;
                if (ct < D) {
                    float add = 0.f;
#pragma unroll
                    for (int g = 0; g < kRowStep; ++g) add += zp[g * D + ct];
                    zreg += add;
                }
                zbuf ^= 1;
            }
            return true;
        };

        auto process_q = [&](int i, int n) -> bool { return q_features(i, n, ct); };


        if (MODE == kApply) {
            // Z rows from the global key sum; then every query item in order
            if (NORM && ct < D) {
                const __nv_bfloat16 h = __float2bfloat16_rn(zreg);
                zr_elem(0, 0, ct) = h;
                zr_elem(0, 1, ct) = __float2bfloat16_rn(zreg - __bfloat162float(h));
            }
            fence_proxy_async();
            for (int n = 0; n < nck * G && ok; ++n) ok = process_q(n / G, n);
        } else {
            // keys of chunk i, then its query heads, chunk after chunk
            for (int i = 0; i < nck && ok; ++i) {
                ok = process_kv(i);
                if (MODE == kCausal && !kQOnEpi)
                    for (int r = 0; r < G && ok; ++r) ok = process_q(i, i * G + r);
            }
            // key sum: final (causal, last segment) or this segment's increment (state pass)
            const bool write_z = ok && nck > 0 && NORM && ct < D && a.Z_dst &&
                                 ((MODE == kCausal && seg == nseg - 1) || MODE == kState);
            if (write_z)
                (MODE == kState ? a.Z_dst + ((size_t)bh * nseg + seg) * D : a.Z_dst + (size_t)bh * D)[ct] = zreg;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, Cf::kTmemCols);
    }
}

}  // namespace chunk
}  // namespace la
