// Balanced split-KV decode over 8-bit caches (head_dim 128, groups of up to 8 query heads).
//
// The method is the split-KV decode's ("TileInfer.jl - Attention kernels", Decode: GQA packing and
// split-KV; "32. Production attention kernels", Long contexts: split the keys): each CTA runs the
// online softmax over a range of keys of one KV head and either writes the normalised rows or an
// unnormalised partial (acc, m, l) that a log-sum-exp combine merges.
//
// What differs is how the keys are cut. The 8-bit consumers stream about 20 GB/s per CTA (their
// per-chunk chain, not HBM, bounds a CTA), and two CTAs fit per SM, so the 64 x 4096 batch's 512
// one-split CTAs run as a full wave of 304 and a second wave two thirds full. Here every CTA that can
// be resident at once gets the same share: the grid is (X, Hkv) with X = resident CTAs / Hkv, every
// KV head's chunks (16 keys) of all sequences are laid end to end, and CTA x streams chunks
// [x C, x C + C), C = ceil(total / X), walking the sequences that range covers (a CTA loops over its
// sequences; the producers keep the ring full across their boundaries). A sequence wholly inside one
// CTA's range is normalised and written there; a sequence cut between CTAs leaves one partial per
// piece, in two slots per CTA (its first and its last sequence), and the combine merges those.
// Every CTA scans the context lengths into chunk offsets in shared memory first.
//
// The per-chunk arithmetic is the split-KV decode's for 8-bit codes: codes straight from the ring
// into fp16 MMA operands, the key scale on the scores, the value scale on the probabilities, int8
// offsets removed after the products.
#include <atomic>

#include "decode_common.cuh"

namespace pa {
namespace {

using namespace dec;

constexpr int kSegD = 128;
constexpr int kSegRows = 8;  // one MMA n-tile of packed query heads
constexpr int kSegMaxUnits = 4096;

template <int QK>
struct SegCfg {
  using C = DecCfg<kSegD, QK>;
  static constexpr int kOffBars = C::kRingBytes;
  static constexpr int kOffScales = kOffBars + 2 * C::kStages * 8;
  static constexpr int kOffMergeMl = kOffScales + C::kStages * 32 * 4;
  static constexpr int kOffMergeO = kOffMergeMl + C::kConsumers * kSegRows * 2 * 4;
  static constexpr int kOffOff = kOffMergeO + C::kConsumers * kSegRows * kSegD * 4;
  static constexpr int kSmemBytes = 1024 + kOffOff + (kSegMaxUnits + 1) * 4;
};

__device__ __forceinline__ int seg_clamped_len(const DecodeParams& p, int u, bool report) {
  const int cap = p.max_blocks * p.block_size;
  int len = p.context_lens[u];
  if (len < 0 || len > cap) {
    if (report) flag_error(p.err, PA_ERRBIT_LENGTH_OUT_OF_RANGE);
    len = len < 0 ? 0 : cap;
  }
  return len;
}
// first position the sequence's query sees (> 0 only under a sliding window)
__device__ __forceinline__ int seg_start(const DecodeParams& p, int len) {
  return p.window > 0 ? max(0, len - p.window) : 0;
}

template <int QK>
__global__ void __launch_bounds__(DecCfg<kSegD, QK>::kThreads)
    decode_seg_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap) {
  using C = DecCfg<kSegD, QK>;
  using L = SegCfg<QK>;
  constexpr int D = kSegD, ROWS = kSegRows;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kOffBars);
  uint64_t* empty = full + C::kStages;
  float* scales = reinterpret_cast<float*>(smem + L::kOffScales);      // [stages][32]
  float* merge_ml = reinterpret_cast<float*>(smem + L::kOffMergeMl);   // [consumers][rows][2]
  float* merge_o = reinterpret_cast<float*>(smem + L::kOffMergeO);     // [consumers][rows][D]
  int* off = reinterpret_cast<int*>(smem + L::kOffOff);                // [units + 1] chunk offsets
  __shared__ int s_timeout;
  __shared__ int s_issued[C::kProducers];
  __shared__ int s_warp_sums[C::kThreads / 32];

  const int x = blockIdx.x, X = gridDim.x, kvh = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.num_units;
  const bool reporter = x == 0 && kvh == 0;
  // the combine launched after this grid may start its launch; it waits for this grid's completion
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
  }

  // ---- chunk counts of the sequences and their exclusive prefix sums (every CTA, in parallel)
  const int per = (S + C::kThreads - 1) / C::kThreads;
  int run = 0;
  for (int k = 0; k < per; ++k) {
    const int u = tid * per + k;
    if (u < S) {
      const int len = seg_clamped_len(p, u, reporter);
      const int c = (len + kChunk - 1) / kChunk - seg_start(p, len) / kChunk;
      off[u] = c;
      run += c;
    }
  }
  int incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_warp_sums[warp] = incl;
  __syncthreads();
  int base = incl - run;
  for (int w = 0; w < warp; ++w) base += s_warp_sums[w];
  for (int k = 0; k < per; ++k) {
    const int u = tid * per + k;
    if (u < S) {
      const int c = off[u];
      off[u] = base;
      base += c;
    }
  }
  if (tid == C::kThreads - 1) off[S] = base;  // the last thread's running sum is the total
  __syncthreads();
  if (reporter)  // the combine reads the offsets from the workspace
    for (int u = tid; u <= S; u += C::kThreads) p.seg_off[u] = off[u];
  const int T = off[S];
  const int Cx = (T + X - 1) / X;
  const int c_lo = min(T, x * Cx), c_hi = min(T, c_lo + Cx);
  if (c_lo >= c_hi) return;  // uniform: no chunks here
  // the sequence holding chunk c_lo: the last u with off[u] <= c_lo (its count is then > 0)
  int u_first = 0;
  {
    int lo = 0, hi = S;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (off[mid] <= c_lo) lo = mid; else hi = mid;
    }
    u_first = lo;
  }
  const int n_mine = c_hi - c_lo;
  if (tid == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&full[i], 33);  // the TMA's expect_tx arrival + the 32 scale-copy arrivals
      mbar_init(&empty[i], 1);
    }
    fence_barrier_init();
    s_timeout = 0;
    for (int w = 0; w < C::kProducers; ++w) s_issued[w] = 0;
  }
  __syncthreads();

  if (warp >= C::kConsumers) {
    // ---------------- producers: chunk i of the range (producer warp i mod kProducers), its
    // sequence found by walking the offsets; page ids fetched 32 at a time per sequence
    const int pw = warp - C::kConsumers;
    int u = u_first, u_lo = off[u], u_hi = off[u + 1];
    int len = seg_clamped_len(p, u, false), cs = seg_start(p, len) / kChunk;
    const int32_t* table = p.block_tables + (size_t)u * p.max_blocks;
    int win_base = -64, my_page = -1;
    int issued = 0;
    for (int i = pw; i < n_mine; i += C::kProducers) {
      const int g = c_lo + i;
      if (g >= u_hi) {  // the next sequence with chunks at or past g
        while (g >= off[u + 1]) ++u;
        u_lo = off[u];
        u_hi = off[u + 1];
        len = seg_clamped_len(p, u, false);
        cs = seg_start(p, len) / kChunk;
        table = p.block_tables + (size_t)u * p.max_blocks;
        win_base = -64;
      }
      const int stage = i % C::kStages;
      bool ok = true;
      if (i >= C::kStages) ok = mbar_wait(&empty[stage], ((i / C::kStages) - 1) & 1);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) {
          flag_error(p.err, PA_ERRBIT_WAIT_TIMEOUT);
          atomicExch(&s_timeout, 1);
        }
        break;
      }
      const int tok = (cs + (g - u_lo)) * kChunk;
      const int page_idx = tok / p.block_size;
      const int in_page = tok - page_idx * p.block_size;
      if (page_idx - win_base >= 32 || page_idx < win_base) {  // uniform
        win_base = page_idx;
        my_page = (win_base + lane < p.max_blocks) ? __ldg(table + win_base + lane) : -1;
      }
      const int page = __shfl_sync(0xffffffffu, my_page, page_idx - win_base);
      const bool page_ok = page >= 0 && page < p.num_blocks;
      {
        // lanes 0-15: the chunk's key scales, 16-31: its value scales, copied asynchronously;
        // positions past the sequence end, or on a page outside the pool, are zero-filled
        const int t = lane & 15;
        const bool take = page_ok && tok + t < len;
        const float* sbase = lane < 16 ? p.k_scales : p.v_scales;
        const float* src = take ? sbase + ((size_t)page * p.block_size + in_page + t) * p.num_kv_heads + kvh : sbase;
        asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_addr(scales + stage * 32 + lane)),
                     "l"(src), "r"(take ? 4 : 0)
                     : "memory");
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(&full[stage]))
                     : "memory");
      }
      if (lane == 0) {
        if (!page_ok) flag_error(p.err, PA_ERRBIT_PAGE_OUT_OF_POOL);  // TMA reads zeros
        uint8_t* st = smem + stage * C::kStageBytes;
        mbar_arrive_expect_tx(&full[stage], C::kStageBytes);
        tma_load_4d(st, &kmap, &full[stage], 0, kvh, in_page, page);
        tma_load_4d(st + C::kTileBytes, &vmap, &full[stage], 0, kvh, in_page, page);
      }
      issued = i + 1;
    }
    if (lane == 0) s_issued[pw] = issued;
  } else {
    // ---------------- consumers: the segments of the range, one sequence each
    const int G = p.group;
    const int g4 = lane >> 2, t4 = lane & 3;
    const int mi = lane >> 3, ri = lane & 7;
    const int k_key = ri + 8 * (mi & 1), k_unit = mi >> 1;
    constexpr int kRegionStride = kChunk * 128;
    const float sl2 = p.scale_log2;
    for (int u = u_first; u < S && off[u] < c_hi; ++u) {
      const int seg_lo = max(off[u], c_lo), seg_hi = min(off[u + 1], c_hi);
      if (seg_hi <= seg_lo) continue;  // a sequence without keys (uniform)
      const int len = seg_clamped_len(p, u, false);
      const int start = seg_start(p, len);
      const int cs = start / kChunk;
      // the sequence's queries: rows n = the G heads of this KV head, fp16, in the codes' k-slot order
      uint32_t qf[C::kMT][2];
      {
        const int n = g4;
        const bool rv = n < G;
        const uint32_t* qr = reinterpret_cast<const uint32_t*>(reinterpret_cast<const __nv_bfloat16*>(p.q) +
                                                               (size_t)u * p.q_stride + (size_t)(kvh * G + (rv ? n : 0)) * D);
#pragma unroll
        for (int kk = 0; kk < C::kMT; ++kk) {
          qf[kk][0] = rv ? bf16x2_to_f16x2(__ldg(qr + (kk * 16 + 4 * t4) / 2)) : 0u;
          qf[kk][1] = rv ? bf16x2_to_f16x2(__ldg(qr + (kk * 16 + 4 * t4 + 2) / 2)) : 0u;
        }
      }
      float qb[2] = {0.f, 0.f};  // int8: 1152 times each score row's query dim sum
      if constexpr (QK == 1) {
        float part = 0.f;
#pragma unroll
        for (int kk = 0; kk < C::kMT; ++kk) {
          const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&qf[kk][0]));
          const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&qf[kk][1]));
          part += (a.x + a.y) + (b.x + b.y);
        }
        part += __shfl_xor_sync(0xffffffffu, part, 1);
        part += __shfl_xor_sync(0xffffffffu, part, 2);
        qb[0] = kCodeBias * __shfl_sync(0xffffffffu, part, 8 * t4);
        qb[1] = kCodeBias * __shfl_sync(0xffffffffu, part, 8 * t4 + 4);
      }
      float o[C::kMT][4];
      float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
      float psum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int mt = 0; mt < C::kMT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
      // this consumer's chunks of the segment: local indices i = warp (mod kConsumers)
      const int i0 = seg_lo - c_lo;
      const int i_first = i0 + (((warp - i0) % C::kConsumers) + C::kConsumers) % C::kConsumers;
      for (int i = i_first; i < seg_hi - c_lo; i += C::kConsumers) {
        const int stage = i % C::kStages;
        if (!mbar_wait(&full[stage], (i / C::kStages) & 1)) {
          flag_error(p.err, PA_ERRBIT_WAIT_TIMEOUT);
          atomicExch(&s_timeout, 1);
          break;
        }
        uint8_t* kt = smem + stage * C::kStageBytes;
        uint8_t* vt = kt + C::kTileBytes;
        const int key0 = (cs + (c_lo + i - off[u])) * kChunk;
        const int nvalid = min(kChunk, len - key0);
        const float* sc = scales + stage * 32;
        const float ks_a = sc[g4], ks_b = sc[g4 + 8], vs_a = sc[16 + g4], vs_b = sc[16 + g4 + 8];
        uint32_t kw[C::kMT][2], vw[C::kMT][2];
        auto load_codes = [&](const uint8_t* tile, uint32_t (&w)[C::kMT][2], bool trans) {
#pragma unroll
          for (int k2 = 0; k2 < C::kMT / 2; ++k2) {
            const uint32_t offb = (k2 >> 2) * kRegionStride + swz128(k_key, 2 * (k2 & 3) + k_unit);
            uint32_t r[4];
            if (trans) ldsm_x4_trans(r, smem_addr(tile + offb)); else ldsm_x4(r, smem_addr(tile + offb));
            w[2 * k2][0] = r[0];
            w[2 * k2][1] = r[1];
            w[2 * k2 + 1][0] = r[2];
            w[2 * k2 + 1][1] = r[3];
          }
        };
        load_codes(kt, kw, false);
        load_codes(vt, vw, true);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);  // the codes are in registers
        if (nvalid < kChunk) {  // value codes of keys past the sequence end become 0
          const uint32_t m0 = (2 * t4 < nvalid ? 0x0000ffffu : 0u) | (2 * t4 + 1 < nvalid ? 0xffff0000u : 0u);
          const uint32_t m1 = (2 * t4 + 8 < nvalid ? 0x0000ffffu : 0u) | (2 * t4 + 9 < nvalid ? 0xffff0000u : 0u);
#pragma unroll
          for (int mt = 0; mt < C::kMT; ++mt) {
            vw[mt][0] &= m0;
            vw[mt][1] &= m1;
          }
        }
        // S^T[16 keys x 8 rows] = K . Q^T (E4M3: two accumulator chains, summed after)
        constexpr int kChains = QK == 2 ? 2 : 1;
        float s[4] = {0.f, 0.f, 0.f, 0.f}, s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < C::kMT; ++kk) {
          uint32_t a[4];
          if constexpr (QK == 1) {
            const uint32_t w0 = kw[kk][0] ^ 0x80808080u, w1 = kw[kk][1] ^ 0x80808080u;
            a[0] = biased2_to_f16x2(w0, kSelB01);
            a[1] = biased2_to_f16x2(w1, kSelB01);
            a[2] = biased2_to_f16x2(w0, kSelB23);
            a[3] = biased2_to_f16x2(w1, kSelB23);
          } else {
            e4m3_halves_to_f16x2(kw[kk][0], a[0], a[2]);
            e4m3_halves_to_f16x2(kw[kk][1], a[1], a[3]);
          }
          mma_cache<QK>(kChains == 2 && (kk & 1) ? s2 : s, a, qf[kk][0], qf[kk][1]);
        }
        if constexpr (kChains == 2) {
#pragma unroll
          for (int e = 0; e < 4; ++e) s[e] += s2[e];
        }
        if constexpr (QK == 1) {
          s[0] -= qb[0];
          s[1] -= qb[1];
          s[2] -= qb[0];
          s[3] -= qb[1];
        }
        s[0] *= ks_a;
        s[1] *= ks_a;
        s[2] *= ks_b;
        s[3] *= ks_b;
        float x0, x1, x2, x3;
        if (p.softcap_log2 > 0.f) {
          x0 = score_log2(p, s[0]);
          x1 = score_log2(p, s[1]);
          x2 = score_log2(p, s[2]);
          x3 = score_log2(p, s[3]);
        } else {
          x0 = s[0] * sl2, x1 = s[1] * sl2, x2 = s[2] * sl2, x3 = s[3] * sl2;
        }
        if (key0 + kChunk > len || key0 < start) {  // the sequence's ends only (uniform)
          const int ka = key0 + g4, kb = ka + 8;
          if (ka >= len || ka < start) x0 = x1 = -INFINITY;
          if (kb >= len || kb < start) x2 = x3 = -INFINITY;
        }
        float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
        for (int offx = 4; offx < 32; offx <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, offx));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, offx));
        }
        const bool up0 = mx0 > m_run[0] + kLazyRescale, up1 = mx1 > m_run[1] + kLazyRescale;
        const float mn0 = up0 ? mx0 : m_run[0], mn1 = up1 ? mx1 : m_run[1];
        const float mu0 = (mn0 == -INFINITY) ? 0.f : mn0, mu1 = (mn1 == -INFINITY) ? 0.f : mn1;
        const float p0 = ex2_ftz(x0 - mu0), p2 = ex2_ftz(x2 - mu0);
        const float p1 = ex2_ftz(x1 - mu1), p3 = ex2_ftz(x3 - mu1);
        if (__any_sync(0xffffffffu, up0 || up1)) {
          const float al0 = up0 ? ex2_ftz(m_run[0] - mu0) : 1.f;
          const float al1 = up1 ? ex2_ftz(m_run[1] - mu1) : 1.f;
          l_run[0] *= al0;
          l_run[1] *= al1;
          if constexpr (QK == 1) {
            psum[0] *= al0;
            psum[1] *= al1;
            psum[2] *= al0;
            psum[3] *= al1;
          }
#pragma unroll
          for (int mt = 0; mt < C::kMT; ++mt) {
            o[mt][0] *= al0;
            o[mt][1] *= al1;
            o[mt][2] *= al0;
            o[mt][3] *= al1;
          }
        }
        l_run[0] += p0 + p2;
        l_run[1] += p1 + p3;
        m_run[0] = mn0;
        m_run[1] = mn1;
        const uint32_t pb0 = movmatrix_trans(pack_f16x2(p0 * vs_a, p1 * vs_a));
        const uint32_t pb1 = movmatrix_trans(pack_f16x2(p2 * vs_b, p3 * vs_b));
#pragma unroll
        for (int mt = 0; mt < C::kMT; ++mt) {
          uint32_t a[4];
          if constexpr (QK == 1) {
            const uint32_t w0 = vw[mt][0] ^ 0x80808080u, w1 = vw[mt][1] ^ 0x80808080u;
            a[0] = biased2_to_f16x2(w0, kSelB02);
            a[1] = biased2_to_f16x2(w0, kSelB13);
            a[2] = biased2_to_f16x2(w1, kSelB02);
            a[3] = biased2_to_f16x2(w1, kSelB13);
          } else {
            a[0] = codes2_to_f16x2<QK>(vw[mt][0], kSelB02);
            a[1] = codes2_to_f16x2<QK>(vw[mt][0], kSelB13);
            a[2] = codes2_to_f16x2<QK>(vw[mt][1], kSelB02);
            a[3] = codes2_to_f16x2<QK>(vw[mt][1], kSelB13);
          }
          mma_cache<QK>(o[mt], a, pb0, pb1);
        }
        if constexpr (QK == 1) {
          const uint32_t ones[4] = {kOnesF16x2, kOnesF16x2, kOnesF16x2, kOnesF16x2};
          mma_16816_f16(psum, ones, pb0, pb1);
        }
      }
      if constexpr (QK == 1) {  // the biased values' offset
#pragma unroll
        for (int mt = 0; mt < C::kMT; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) o[mt][e] -= kCodeBias * psum[e];
      }
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int offx = 4; offx < 32; offx <<= 1) l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], offx);
      // merge the four consumers' states: the previous segment's merge has been read by everyone
      // once all consumers pass the first barrier, the states are in place after the second
      asm volatile("bar.sync 1, %0;" ::"n"(C::kConsumers * 32));
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int n = 2 * t4 + j;
        if (g4 == 0) {
          merge_ml[(warp * ROWS + n) * 2] = m_run[j];
          merge_ml[(warp * ROWS + n) * 2 + 1] = l_run[j];
        }
#pragma unroll
        for (int mt = 0; mt < C::kMT; ++mt) {  // accumulator rows g, g+8: dims 2g, 2g+1 of the block
          merge_o[(warp * ROWS + n) * D + mt * 16 + 2 * g4] = o[mt][j];
          merge_o[(warp * ROWS + n) * D + mt * 16 + 2 * g4 + 1] = o[mt][2 + j];
        }
      }
      asm volatile("bar.sync 1, %0;" ::"n"(C::kConsumers * 32));
      // the whole sequence here: normalised rows; else this piece's partial, in this CTA's slot 0
      // (the sequence it starts in) or slot 1 (the one it ends in)
      const bool whole = off[u] >= c_lo && off[u + 1] <= c_hi;
      const size_t slot0 = ((size_t)(x * p.num_kv_heads + kvh) * 2 + (off[u] <= c_lo ? 0 : 1)) * G;
      for (int idx = tid; idx < G * D; idx += C::kConsumers * 32) {
        const int n = idx / D, d = idx - n * D;
        const int h = kvh * G + n;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::kConsumers; ++w) M = fmaxf(M, merge_ml[(w * ROWS + n) * 2]);
        const float Mu = (M == -INFINITY) ? 0.f : M;
        float Lsum = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < C::kConsumers; ++w) {
          const float wt = exp2f(merge_ml[(w * ROWS + n) * 2] - Mu);
          Lsum += wt * merge_ml[(w * ROWS + n) * 2 + 1];
          O += wt * merge_o[(w * ROWS + n) * D + d];
        }
        if (whole) {
          if (p.sinks != nullptr) O *= fold_sink(p.sinks[h], M, Lsum);
          const float v = (Lsum > 0.f) ? O / Lsum : 0.f;
          reinterpret_cast<__nv_bfloat16*>(p.out)[(size_t)u * p.out_stride + (size_t)h * D + d] = __float2bfloat16(v);
        } else {
          p.ws_acc[(slot0 + n) * D + d] = O;
          if (d == 0) {
            p.ws_ml[(slot0 + n) * 2] = M;
            p.ws_ml[(slot0 + n) * 2 + 1] = Lsum;
          }
        }
      }
      if (*reinterpret_cast<volatile int*>(&s_timeout)) break;  // the same verdict in every consumer
    }
  }
  __syncthreads();
  if (s_timeout && threadIdx.x == C::kConsumers * 32) {
    // wind down: let copies still in flight land before the CTA's shared memory is released
    int hi = 0;
    for (int w = 0; w < C::kProducers; ++w) hi = max(hi, s_issued[w]);
    for (int i = max(0, hi - C::kStages); i < hi; ++i)
      if (i < s_issued[i % C::kProducers]) (void)mbar_wait(&full[i % C::kStages], (i / C::kStages) & 1);
  }
  __syncthreads();
}

// Log-sum-exp merge of the pieces of the sequences that were cut between CTAs ("32. Production
// attention kernels", Long contexts: split the keys: M = max m_s, w_s = 2^(m_s - M),
// out = sum w_s acc_s / sum w_s l_s); one warp per (sequence, query head), lanes over head dims.
// Sequences written whole by the decode grid are skipped; sequences without keys get zeros.
__global__ void __launch_bounds__(128) combine_seg_kernel(const __grid_constant__ DecodeParams p) {
  const int gw = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (gw >= p.num_units * p.num_q_heads) return;
  asm volatile("griddepcontrol.wait;" ::: "memory");  // the decode grid's partials and offsets
  const int u = gw / p.num_q_heads, h = gw - u * p.num_q_heads;
  const int G = p.group, kvh = h / G, n = h - kvh * G;
  const int S = p.num_units, X = p.seg_ctas;
  const int T = p.seg_off[S];
  const int o_lo = p.seg_off[u], o_hi = p.seg_off[u + 1];
  __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(p.out) + (size_t)u * p.out_stride + (size_t)h * kSegD;
  const int d = lane * 4;
  if (o_hi <= o_lo) {  // no keys: zeros
    *reinterpret_cast<uint2*>(out + d) = make_uint2(0u, 0u);
    return;
  }
  const int Cx = (T + X - 1) / X;
  const int x1 = o_lo / Cx, x2 = (o_hi - 1) / Cx;
  if (x1 == x2) return;  // written whole by its CTA
  auto slot_of = [&](int x) {
    return ((size_t)(x * p.num_kv_heads + kvh) * 2 + (o_lo <= x * Cx ? 0 : 1)) * G + n;
  };
  float M = -INFINITY;
  for (int x = x1; x <= x2; ++x) M = fmaxf(M, p.ws_ml[slot_of(x) * 2]);
  const float Mu = (M == -INFINITY) ? 0.f : M;
  float Lsum = 0.f;
  float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int x = x1; x <= x2; ++x) {
    const size_t sl = slot_of(x);
    const float w = exp2f(p.ws_ml[sl * 2] - Mu);
    Lsum += w * p.ws_ml[sl * 2 + 1];
    const float4 a = *reinterpret_cast<const float4*>(p.ws_acc + sl * kSegD + d);
    O.x += w * a.x;
    O.y += w * a.y;
    O.z += w * a.z;
    O.w += w * a.w;
  }
  float f = 1.f;
  if (p.sinks != nullptr) f = fold_sink(p.sinks[h], M, Lsum);
  const float inv = (Lsum > 0.f) ? f / Lsum : 0.f;
  uint2 r;
  r.x = pack_bf16x2(O.x * inv, O.y * inv);
  r.y = pack_bf16x2(O.z * inv, O.w * inv);
  *reinterpret_cast<uint2*>(out + d) = r;
}

template <int QK>
int seg_ctas_per_sm() {
  // the occupancy of a kernel above 48 KiB of dynamic shared memory counts only once it may use it
  if (cudaFuncSetAttribute(decode_seg_kernel<QK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           SegCfg<QK>::kSmemBytes) != cudaSuccess)
    return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_seg_kernel<QK>, DecCfg<kSegD, QK>::kThreads,
                                                    SegCfg<QK>::kSmemBytes) != cudaSuccess)
    return 1;
  return n < 1 ? 1 : n;
}

template <int QK>
cudaError_t launch_seg_impl(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                            cudaStream_t stream) {
  static std::atomic<bool> attr_done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_done[dev].load(std::memory_order_acquire)) {
    cudaError_t e = cudaFuncSetAttribute(decode_seg_kernel<QK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SegCfg<QK>::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev].store(true, std::memory_order_release);
  }
  decode_seg_kernel<QK><<<dim3((unsigned)p.seg_ctas, (unsigned)p.num_kv_heads), DecCfg<kSegD, QK>::kThreads,
                          SegCfg<QK>::kSmemBytes, stream>>>(p, kmap, vmap);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const unsigned blocks = (unsigned)(((long long)p.num_units * p.num_q_heads + 3) / 4);
  return launch_dependent(combine_seg_kernel, blocks, 128u, 0, stream, p);
}

}  // namespace

bool decode_seg_supported(int head_dim, int group, int num_units, int quant) {
  return quant != 0 && head_dim == kSegD && group >= 1 && group <= kSegRows && num_units >= 1 &&
         num_units <= kSegMaxUnits;
}

int decode_seg_ctas_per_sm(int quant) {
  static std::atomic<int> occ[64][2] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return quant == 1 ? seg_ctas_per_sm<1>() : seg_ctas_per_sm<2>();
  std::atomic<int>& slot = occ[dev][quant == 1 ? 0 : 1];
  int v = slot.load(std::memory_order_relaxed);
  if (v == 0) {
    v = quant == 1 ? seg_ctas_per_sm<1>() : seg_ctas_per_sm<2>();
    slot.store(v, std::memory_order_relaxed);
  }
  return v;
}

size_t decode_seg_workspace_bytes(int num_units, int num_q_heads, int ctas_per_head) {
  // two partial slots per CTA and query head (acc [D] and (m, l)), then the chunk offsets
  const size_t slots = (size_t)ctas_per_head * 2 * num_q_heads;
  return slots * ((size_t)kSegD + 2) * 4 + ((size_t)num_units + 1) * 4;
}

cudaError_t launch_decode_seg(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                              cudaStream_t stream) {
  return p.quant == 1 ? launch_seg_impl<1>(p, kmap, vmap, stream) : launch_seg_impl<2>(p, kmap, vmap, stream);
}

}  // namespace pa
