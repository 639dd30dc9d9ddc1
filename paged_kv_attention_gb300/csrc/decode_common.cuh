// Device helpers of the decode kernels, shared by the split-KV decode (decode.cu) and its
// balanced-segment form for 8-bit caches (decode_seg.cu): unit resolution, the epilogue merge,
// mma.sync / ldmatrix / movmatrix wrappers, the ring configuration and the 8-bit code conversions.
#pragma once

#include <cuda_fp16.h>

#include "pa_common.cuh"
#include "pa_internal.h"

// Producer warps per decode CTA (measured at 64x4096 on GB300: one producer warp cannot issue
// the page walk's copies as fast as HBM delivers them; 2 for bf16 took the call from 187 to 171 us,
// 4 for 8-bit codes from 194 to 161 us; more warps cost occupancy)
#ifndef PA_DECODE_PRODUCERS_BF16
#define PA_DECODE_PRODUCERS_BF16 2
#endif
#ifndef PA_DECODE_PRODUCERS_CODES
#define PA_DECODE_PRODUCERS_CODES 4
#endif

namespace pa {
namespace dec {


// ------------------------------------------------------------------ unit resolution
struct Unit {
  int len;        // keys [start, len) are loaded; the unit's last query sees all of them
  int start;      // first position any query of the unit sees (> 0 only under a sliding window)
  int table_row;  // block table row
  int q_row;      // row of q / out of the unit's first query
  int n_tok;      // queries of the unit (consecutive rows of q); its rows are n_tok * group
  int first_pos;  // position of the unit's first query; query t sits at first_pos + t
  bool skip;      // not this launch's unit: write nothing
};

__device__ __forceinline__ Unit resolve_unit(const DecodeParams& p, int unit, bool report) {
  Unit u;
  u.skip = false;
  u.n_tok = 1;
  u.first_pos = 0;
  int len;
  if (p.varlen == 0) {
    u.table_row = unit;
    u.q_row = unit;
    len = p.context_lens[unit];
    u.start = 0;
  } else if (p.varlen == 2) {
    // request units: a request with 1 <= q_len <= small_max, its queries in groups of
    // unit_tokens (group g of request r is unit r * groups_per_req + g); every other request is
    // left to the tensor-core kernel and nothing is written for it here
    const int r = unit / p.groups_per_req;
    const int g = unit - r * p.groups_per_req;
    const int start = p.query_start_loc[r];
    const int q_len = p.query_start_loc[r + 1] - start;
    const int tok0 = g * p.unit_tokens;
    u.table_row = r;
    u.start = 0;
    u.q_row = start + tok0;
    if (start < 0 || q_len < 1 || q_len > p.small_max || tok0 >= q_len || start + q_len > p.num_tokens) {
      u.skip = true;  // (a query block past the last row is flagged by the tensor-core kernel)
      len = 0;
    } else {
      u.n_tok = min(p.unit_tokens, q_len - tok0);
      const int seq = p.seq_lens[r];
      if (q_len > seq) {  // the queries' own positions are not all cached: a layout error, zero rows
        if (report) flag_error(p.err, PA_ERRBIT_QUERY_LAYOUT);
        len = 0;
      } else if (seq > p.max_blocks * p.block_size) {  // as the varlen kernels: zero rows, flag
        if (report) flag_error(p.err, PA_ERRBIT_LENGTH_OUT_OF_RANGE);
        len = 0;
      } else {
        u.first_pos = seq - q_len + tok0;  // queries are the request's newest positions
        len = p.causal ? u.first_pos + u.n_tok : seq;
        if (p.window > 0) u.start = max(0, u.first_pos - p.window + 1);
      }
    }
  } else {
    // request r with query_start_loc[r] <= unit < query_start_loc[r+1]
    int lo = 0, hi = p.num_reqs;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (p.query_start_loc[mid] <= unit) lo = mid; else hi = mid;
    }
    const int start = p.query_start_loc[lo];
    const int stop = p.query_start_loc[lo + 1];
    const int seq = p.seq_lens[lo];
    const int q_len = stop - start;
    u.table_row = lo;
    u.q_row = unit;
    u.start = 0;
    if (unit < start || unit >= stop || q_len > seq) {
      if (report) flag_error(p.err, PA_ERRBIT_QUERY_LAYOUT);
      len = 0;
    } else if (seq > p.max_blocks * p.block_size) {
      if (report) flag_error(p.err, PA_ERRBIT_LENGTH_OUT_OF_RANGE);
      len = 0;
    } else {
      const int pos = seq - q_len + (unit - start);  // queries are the newest positions
      len = p.causal ? pos + 1 : seq;
      u.first_pos = pos;
      if (p.window > 0) u.start = max(0, pos - p.window + 1);
    }
  }
  const int cap = p.max_blocks * p.block_size;
  if (len < 0 || len > cap) {
    if (report) flag_error(p.err, PA_ERRBIT_LENGTH_OUT_OF_RANGE);
    len = len < 0 ? 0 : cap;
  }
  u.len = len;
  if (p.varlen == 0) {
    // decode: the query is the newest cached position, len - 1
    u.first_pos = len - 1;
    if (p.window > 0) u.start = max(0, len - p.window);
  }
  if (u.start > u.len) u.start = u.len;
  return u;
}

// Threshold of the lazy rescale (log2 units): probabilities against a stale reference are < 2^8.
constexpr float kLazyRescale = 8.0f;

// Score in log2 units: s * scale * log2 e, or with a softcap c: c * tanh(s * scale / c) * log2 e
// ("poot - Attention and KV Cache", The streaming schedule: softcap_or_identity).
__device__ __forceinline__ float score_log2(const DecodeParams& p, float s) {
  return p.softcap_log2 > 0.f ? p.softcap_log2 * tanhf(s * p.scale_over_cap) : s * p.scale_log2;
}

// ------------------------------------------------------------------ epilogue
// Merge the per-warp online-softmax states kept in shared memory and write either the
// normalised rows (one split) or this split's unnormalised partial.
//   mo: [nw][rows][D] accumulators, ml: [nw][rows][2] (m in log2 units, l)
template <typename OutT>
__device__ __forceinline__ void merge_and_store(const DecodeParams& p, const float* mo, const float* ml, int nw,
                                                int rows, int D, int unit, const Unit& u, int kvh, int split) {
  const int G = p.group;
  // row n of the state: query t = n / G of the unit, head kvh * G + n % G
  for (int idx = threadIdx.x; idx < u.n_tok * G * D; idx += blockDim.x) {
    const int n = idx / D;
    const int d = idx - n * D;
    const int t = n / G;
    const int h = kvh * G + (n - t * G);
    float M = -INFINITY;
    for (int w = 0; w < nw; ++w) M = fmaxf(M, ml[(w * rows + n) * 2]);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float L = 0.f, O = 0.f;
    for (int w = 0; w < nw; ++w) {
      const float wt = exp2f(ml[(w * rows + n) * 2] - Mu);
      L += wt * ml[(w * rows + n) * 2 + 1];
      O += wt * mo[(w * rows + n) * D + d];
    }
    if (p.num_splits == 1 && !p.force_partial) {
      if (p.sinks != nullptr) O *= fold_sink(p.sinks[h], M, L);
      const float v = (L > 0.f) ? O / L : 0.f;
      OutT* out = reinterpret_cast<OutT*>(p.out);
      out[(size_t)(u.q_row + t) * p.out_stride + (size_t)h * D + d] = static_cast<OutT>(v);
    } else {
      // partial slot (unit, split, query t of the unit, head)
      const size_t slot =
          (((size_t)unit * p.slot_count + p.slot_offset + split) * p.unit_tokens + t) * p.num_q_heads + h;
      p.ws_acc[slot * D + d] = O;
      if (d == 0) {
        p.ws_ml[slot * 2] = M;
        p.ws_ml[slot * 2 + 1] = L;
      }
    }
  }
}

// ------------------------------------------------------------------ bf16 tensor-core decode
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_16816_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// bf16 operands for bf16 caches, fp16 for converted 8-bit codes
template <int QK>
__device__ __forceinline__ void mma_cache(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  if constexpr (QK == 0) mma_16816(c, a, b0, b1); else mma_16816_f16(c, a, b0, b1);
}
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// QK selects the cache format: 0 = bf16 values; 1 = int8 codes, 2 = fp8 E4M3 codes, each with
// one fp32 scale per (slot, KV head). 8-bit codes go from the ring straight into MMA operand
// registers (ldmatrix over byte pairs) and are converted there, exactly, to fp16; the key's scale
// multiplies its scores and the value's scale its probabilities before P.V ("TileInfer.jl -
// Attention kernels", INT8 cache). The page converts to bf16; here the 16-bit type is fp16, which
// holds every code exactly, so the MMAs for 8-bit caches run in fp16 with fp32 accumulation, the
// queries converted once per CTA (exact within fp16's range) and the probabilities rounded to fp16
// (3 more mantissa bits than bf16). An int8 code c becomes the fp16 1152 + c with one byte permute
// per two codes; the MMAs take the offset codes and the 1152 offsets are taken out of their sums
// afterwards (exact up to fp32 rounding of sums some 1152 times larger than the codes'). E4M3
// codes take one conversion instruction per pair.
//
// Register-direct operands rest on two permutations the products do not see. Scores: an
// ldmatrix of byte pairs hands a thread 4 consecutive codes of a key row, so the k-slots
// (2t, 2t+1 | 2t+8, 2t+9) of the m16n8k16 A fragment hold head dims (4t, 4t+1 | 4t+2, 4t+3) of
// each 16-dim step, and the queries are loaded with the same order (a dot product is invariant
// under a common permutation of its terms). P.V: a transposing ldmatrix hands a thread keys
// (2t, 2t+1) of the dim pair (2g, 2g+1), so A rows g and g+8 of each 16-dim block are head dims
// 2g and 2g+1; the accumulator rows are written back to those dims.
template <int D, int QK>
struct DecCfg {
  static constexpr int kConsumers = 4;
  // producer warps take the chunks in turn
  static constexpr int kProducers = QK ? PA_DECODE_PRODUCERS_CODES : PA_DECODE_PRODUCERS_BF16;
  static constexpr int kThreads = (kConsumers + kProducers) * 32;
  static constexpr int kElt = QK ? 1 : 2;                // bytes per cached element
  static constexpr int kBoxes = D * kElt / 128;          // 128-byte swizzle columns of a cached row
  static constexpr int kTileBytes = kChunk * D * kElt;   // K or V rows of one stage
  static constexpr int kStageBytes = 2 * kTileBytes;
  // a 64 KiB ring: 8 stages of 8 KiB for bf16 at D 128; 16 stages of 4 KiB for codes at D 128
  static constexpr int kStages = 65536 / kStageBytes;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kMT = D / 16;
  static constexpr int kScaleBytes = QK ? kStages * 32 * 4 : 0;                   // 16 K + 16 V scales per stage
  // ring | full, empty barriers | merge (m, l) | scales; the merge accumulators alias the ring
  static constexpr int kSmemBytes = 1024 + kRingBytes + 2 * kStages * 8 + kConsumers * 16 * 2 * 4 + kScaleBytes;
  static_assert(kBoxes >= 1, "a cached row must span at least one 128-byte column");
  static_assert(kStages % kConsumers == 0, "stages are dealt to consumers round robin");
  // each stage must always be refilled by the same producer warp, so that it waits on the
  // stage's "empty" phases in order: a parity wait cannot tell phase j from phase j - 2, and a
  // producer running a ring lap ahead of another would take a stage still in use
  static_assert(kStages % kProducers == 0, "stages are dealt to producers round robin");
  static_assert(kConsumers * 16 * D * 4 <= kRingBytes, "merge area must fit in the ring");
};

// Two codes of a 4-code word (bytes `sel` picks: byte 0 and byte 1 of the selector's low nibbles)
// -> an fp16 pair, exactly (|int8 code| <= 128 and every E4M3 value are fp16 values).
// int8: code c -> byte c + 128 -> the fp16 with bits 0x64bb is 1024 + b, so subtracting 1152
// leaves c: one byte permute and one packed subtraction per two codes.
template <int QK>
__device__ __forceinline__ uint32_t codes2_to_f16x2(uint32_t w, uint32_t sel) {
  if constexpr (QK == 1) {
    const uint32_t h = __byte_perm(w ^ 0x80808080u, 0x64646464u, sel);
    const __half2 c = __hsub2(*reinterpret_cast<const __half2*>(&h), __half2half2(__ushort_as_half(0x6480)));
    return *reinterpret_cast<const uint32_t*>(&c);
  } else {
    // the same two bytes, packed into the low half-word, through the E4M3 -> f16x2 conversion
    const uint32_t pair = __byte_perm(w, 0u, (sel & 0xfu) | ((sel & 0xf00u) >> 4));
    uint32_t h;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"((unsigned short)pair));
    return h;
  }
}
// int8 without the subtraction: two codes of a word already flipped to c + 128 (w ^ 0x80808080)
// -> the fp16 pair 1152 + c, exactly; one byte permute per two codes. The consumers remove the
// 1152 offsets after the products: from the scores with the query's dim sum (once per CTA), from
// P.V with the probability sums that one more MMA against an all-ones operand accumulates.
__device__ __forceinline__ uint32_t biased2_to_f16x2(uint32_t flipped, uint32_t sel) {
  return __byte_perm(flipped, 0x64646464u, sel);
}
constexpr float kCodeBias = 1152.f;
constexpr uint32_t kOnesF16x2 = 0x3c003c00u;  // fp16 (1, 1)
// E4M3: the two code pairs of a word in adjacent bytes (0-1 and 2-3), each a 16-bit half of the
// word, converted without a byte permute
__device__ __forceinline__ void e4m3_halves_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}
// selectors (result bytes 0 and 2 carry the codes; bytes 1 and 3 take 0x64 from the constant)
constexpr uint32_t kSelB01 = 0x5140;  // codes in bytes 0, 1
constexpr uint32_t kSelB23 = 0x5342;  // codes in bytes 2, 3
constexpr uint32_t kSelB02 = 0x5240;  // codes in bytes 0, 2
constexpr uint32_t kSelB13 = 0x5341;  // codes in bytes 1, 3

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 v = __floats2half2_rn(lo, hi);  // .x = lo (low half)
  return *reinterpret_cast<const uint32_t*>(&v);
}

// bf16 pair -> fp16 pair (exact within fp16's range)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t v) {
  const float lo = __uint_as_float(v << 16), hi = __uint_as_float(v & 0xffff0000u);
  return pack_f16x2(lo, hi);
}

}  // namespace dec
}  // namespace pa
