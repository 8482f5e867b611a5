// Split-KV absorbed decode on the fifth-generation tensor cores (128 heads,
// the DeepSeek-V3 shape), bf16 latent cache.
//
// What it computes (per worker range of 64-token pages, see decode_plan.cu),
// following "DeepSeek MLA 吸收式缓存" §2.2–§2.4 and §6.1 (MQA over the latent:
// key width 576, value width 512):
//   S[h,t] = q_lat[h] . c_t + q_pe[h] . k_pe_t          (M = 128 heads, K = 576)
//   online softmax over t (log2 domain, scale folded in)
//   O[h,:] += P[h,t] c_t                                (M = 128, N = 512)
//   emitted per segment as O / l (rounded to bf16) and LSE = (m + log2 l) ln 2.
//
// Why a CTA pair.  O is 128 x 512 fp32 = 256 KB, all of one SM's tensor memory.
// The pair splits the latent width: CTA r owns latent dims [256r, 256r+256)
// and RoPE dims [32r, 32r+32), TMA-loads only that half of every 64-token page
// (HBM bytes are not duplicated), and accumulates its O half (128 x 256 fp32,
// TMEM) += P . V_half.  A score needs both halves of the width, so the pair
// splits the softmax by token: CTA r runs the softmax of all 128 heads over
// tokens [32r, 32r+32) of every page ("my" tokens).  Per page each CTA
//  * computes its partial S (M=128 heads, N=64 tokens, K=288) into TMEM, with
//    its half of q_lat in TMEM and its half of q_pe in shared memory as A
//    operands;
//  * sends the peer the partial scores of the peer's 32 tokens, already in log2
//    units, as fp16 (8 KB: each lane-quadrant warp writes its 32 heads' rows to
//    a local staging tile and ships them, 2 KB, with one bulk shared-to-peer
//    copy counted on the peer's transaction barrier of that quadrant);
//  * adds the peer's partial to its own for my tokens, forms P = 2^(s - m_ref)
//    in bf16 for those 32 columns (two 16-token tiles of its P) and ships them
//    (each softmax warp its own 1 KB of rows) with a per-head message (its
//    slice maximum, or its slice sum at a segment end);
//  * issues O_half += P . V_half as soon as both token halves of P are in
//    place: one transaction barrier counts the local warps' P and the peer's
//    8 KB, so a page's P.V waits for nothing else.
// Distributed shared memory moves ~14.5 bytes per cycle per SM each way, less
// than the ~23 bytes per cycle per SM that HBM delivers, so the 17 KB per page
// each way (against 36 KB of cache streamed) is the design's budget: fp32
// partials (32 KB) would cap the kernel well below the HBM roofline.
//
// The reference maximum.  Both CTAs must write P in the same reference m_ref
// (their halves feed one accumulator).  At a segment's first page the pair
// swaps its slice maxima and both take the exact maximum.  Later pages use the
// running reference; at the end of the next page, when all four slice
// messages of a page have arrived, both CTAs move the reference if the page
// maximum exceeded it by more than 2^8: the P of the pages written so far is
// already in the old reference, so O is rescaled by the same factor on both
// sides once the last of those pages' P.V has completed, before the next
// page's P.V (which needs this CTA's next P).  A score more than 2^100 above
// its reference cannot be weighted exactly in that reference: p is capped
// there (O and l stay finite) and the row is flagged in the plan block, and the
// combine kernel recomputes the flagged rows with a plain online softmax that
// rescales at every new maximum.  So does a row whose exchanged fp16 half
// scores exceed 2^5 in magnitude (beyond it an fp16 half score carries more
// than 2^-7 of absolute error, 0.5 % on p).
//
// MMA issue.  A tcgen05.mma blocks its issuing thread while an MMA on the same
// accumulator is in flight, so three threads issue MMAs: S of even pages, S of
// odd pages (two score buffers in TMEM), and P.V (O).  The P.V completion is
// signalled to both CTAs (multicast commit): a P tile is rewritten only once
// both CTAs' P.V have read it.
//
// Warp roles (512 threads): warps 0..3 are the TMA producer, the P.V issuer
// and the two S issuers (even / odd pages), assigned per rank; warp 1 owns
// TMEM.  TMEM lane quadrant q = warp % 4 holds heads 32q..32q+31 and is served
// by three softmax warps: two "MT" warps own 16 of my tokens each (and 128
// columns each of O), one "PT" warp ships the partial scores of the peer's
// tokens and, for quantized pools, dequantizes the page two ahead.  Exchange
// buffers and barriers are per lane quadrant, so the page loop has no
// group-wide barrier.  Every wait is bounded; its polling loop is out of line
// (most waits end at the first probe, and the kernel's code must stay small:
// instruction fetch is on the per-page chain).  A timeout records
// MLA_ERR_TIMEOUT, raises the abort flag of both CTAs, lets in-flight copies
// and MMAs land, frees TMEM and returns.
//
// Tensor memory (512 columns): O [0,256), q_lat half [256,384), S double
// buffer [384,512).
#include <cstddef>
#include <cstring>
#include <mutex>

#include "tc_ptx.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr int TC_THREADS = 512;  // 4 role warps + per TMEM lane quadrant 2 MT warps and 1 PT warp
constexpr int SOFT_WARP0 = 4;
constexpr int TILE = 64;                                      // tokens per page / TMA stage / S tile
constexpr int HALF_C = 256;
constexpr int PE_HALF = 32;
constexpr int HALF_T = 32;                                    // tokens of a page whose softmax one CTA runs
constexpr int TPW = 16;                                       // tokens of a page per MT thread
constexpr int QCOLS = 64;                                     // q_lat TMEM columns (bf16 pairs) per MT thread
constexpr uint32_t KV_CHUNK = TILE * 64 * 2;                  // 8,192: [64 tokens][64 dims] 128B-swizzled
constexpr uint32_t KV_PE_OFF = 4 * KV_CHUNK;                  // 32,768: [64 tokens][32 dims] 64B-swizzled
constexpr uint32_t KV_BYTES = TILE * (HALF_C + PE_HALF) * 2;  // 36,864
constexpr uint32_t PG_BYTES = 128 * TPW * 2;                  // 4,096: P of 16 tokens, [128][16] 32B-swizzled
constexpr uint32_t X_BYTES = 128 * HALF_T * 2;                // 8,192: fp16 partial scores of a token half
constexpr uint32_t X_Q = X_BYTES / 4;                         // 2,048: the rows of one TMEM lane quadrant
constexpr uint32_t PG_Q = PG_BYTES / 4;                       // 1,024: one MT warp's rows of its P tile
constexpr uint32_t SL_Q = 32 * 4;                             // 128: one MT warp's message (a float per head)
constexpr uint32_t PIN_Q = 2 * SL_Q;                          // messages from the peer's two MT warps of a quadrant
constexpr uint32_t QPE_BYTES = 128 * PE_HALF * 2;             // 8,192: [128 heads][32 dims] 64B-swizzled
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_O = 0, TM_Q = 256, TM_S = 384;
constexpr int Q_AHEAD = 8;  // pages before a row's end at which the producer prefetches the next query
constexpr uint32_t QT_BYTES = 128 * 64 * 2;  // 16,384: one q_lat tile, [128 heads][64 dims] 128B-swizzled
constexpr float RESCALE_LOG2 = 8.f;  // move the running max only when it grows by > 2^8
constexpr float RANGE_LOG2 = 100.f;  // largest exponent of p formed here (O and l stay finite in fp32)
constexpr float EXCH_LOG2 = 32.f;    // largest |half score| (log2 units) exchanged in fp16 for an exact row
constexpr long long WAIT_LIMIT_CYCLES = 4000000000ll;  // ~2 s at the maximum SM clock

// Per cache format: bf16 pages are TMA-copied straight into the MMA operand
// stages (4 of them).  Quantized pages land in a small staging ring of codes
// and scales; the sender warps dequantize each into a bf16 operand stage (3 of
// them, and a single staging tile for the shipped partial scores: shared
// memory holds no more next to the staging ring).  Offsets are
// bytes inside one staging slot (this CTA's half of a page, unswizzled rows):
//   INT8: c codes i8 [64][256] | k_pe codes i8 [64][32] | c scales bf16 [64][8]
//         | k_pe scales bf16 [64][8] (all 8 groups of the token)
//   INT4: c codes u8 [64][128] (2 per byte) | k_pe codes i8 [64][32] | c scales
//         bf16 [64][8] | c zeros bf16 [64][8] | k_pe scales bf16 [64][8]
template <int FMT> struct FmtTraits;
template <> struct FmtTraits<MLA_FMT_BF16> {
  static constexpr int KV_ST = 4, CODE_ST = 0;
  static constexpr uint32_t CODE_BYTES = 0, C_OFF = 0, PE_OFF = 0, CS_OFF = 0, ZS_OFF = 0, PS_OFF = 0;
};
template <> struct FmtTraits<MLA_FMT_INT8> {
  static constexpr int KV_ST = 3, CODE_ST = 2;
  static constexpr uint32_t C_OFF = 0, PE_OFF = 16384, CS_OFF = 18432, ZS_OFF = 0, PS_OFF = 19456;
  static constexpr uint32_t CODE_BYTES = 20480;
};
template <> struct FmtTraits<MLA_FMT_INT4> {
  static constexpr int KV_ST = 3, CODE_ST = 3;
  static constexpr uint32_t C_OFF = 0, PE_OFF = 8192, CS_OFF = 10240, ZS_OFF = 11264, PS_OFF = 12288;
  static constexpr uint32_t CODE_BYTES = 13312;
};

template <int FMT>
struct __align__(1024) SmemTC {
  static constexpr int KV_ST = FmtTraits<FMT>::KV_ST;
  static constexpr int CODE_ST = FmtTraits<FMT>::CODE_ST > 0 ? FmtTraits<FMT>::CODE_ST : 1;
  static constexpr uint32_t CODE_BYTES = FmtTraits<FMT>::CODE_BYTES > 0 ? FmtTraits<FMT>::CODE_BYTES : 128;
  uint8_t kv[KV_ST][KV_BYTES];
  uint8_t qpe[QPE_BYTES];     // 64B-swizzled MMA operand: 1 KB aligned (follows 1 KB multiples)
  uint8_t p[2][4][PG_BYTES];  // P per page parity and 16-token group ([128 heads][16 tokens], 32B-swizzled)
  uint8_t xin[2][X_BYTES];    // the peer's fp16 partials of our token half, rows 64 B, chunks swizzled
  static constexpr int XOUT_N = FMT == MLA_FMT_BF16 ? 2 : 1;
  uint8_t xout[XOUT_N][X_BYTES];  // ours of the peer's token half, same layout, shipped by one bulk copy
  uint8_t code[CODE_ST][CODE_BYTES];  // quantized formats: staged codes and scales of a page half
  // per page (mod 4), slice (2 rank + MT index) and head: the slice maximum
  // (its sum at a segment end), ours written here and shipped, the peer's
  // copied in.  Four pages deep: a check reads page j's one page later, and
  // page j+4's arrive only after this CTA's P of page j+2, which comes after
  // that check in every MT warp.  mxs: a segment's first-page slice maxima
  // (bf16: both CTAs take the reference from the same rounded values),
  // exchanged before its P; rewritten at the next segment start only after
  // all four MT warps of the quadrant have read them (mx_empty)
  float msgs[4][4][128];
  uint16_t mxs[4][128];
  uint64_t kv_full[KV_ST], kv_empty[KV_ST];
  uint64_t code_full[CODE_ST], code_empty[CODE_ST];
  uint64_t q_ready;         // quantized: q_lat half in TMEM (8 warp arrivals) + q_pe half in smem (1 arrival + bytes)
  uint64_t q_done, qpe_full;  // bf16: the segment's q_lat half copied into TMEM / its q_pe half into qpe
  uint64_t s_full[2], s_free[2];
  uint64_t p_full[2], pv_done[2], pv_both[2];
  uint64_t x_full[2][4], x_empty[2][4], pin_full[2][4];  // per page parity and lane quadrant
  uint64_t mx_full[4], mx_empty[4];  // per lane quadrant, one phase per segment start
  uint64_t o_free, mma_done[3];
  uint32_t tmem_base;
  volatile int abort_flag;
};
static_assert(sizeof(SmemTC<MLA_FMT_BF16>) + 1024 <= 232448, "shared memory of one CTA exceeds 227 KB");
static_assert(sizeof(SmemTC<MLA_FMT_INT8>) + 1024 <= 232448, "shared memory of one CTA exceeds 227 KB");
static_assert(sizeof(SmemTC<MLA_FMT_INT4>) + 1024 <= 232448, "shared memory of one CTA exceeds 227 KB");
static_assert(KV_BYTES % 1024 == 0 && PG_BYTES % 1024 == 0 && QPE_BYTES % 1024 == 0,
              "swizzled tiles need 1 KB alignment");
static_assert(offsetof(SmemTC<MLA_FMT_BF16>, qpe) % 1024 == 0 && offsetof(SmemTC<MLA_FMT_BF16>, p) % 1024 == 0 &&
                  offsetof(SmemTC<MLA_FMT_INT8>, qpe) % 1024 == 0 && offsetof(SmemTC<MLA_FMT_INT4>, qpe) % 1024 == 0,
              "swizzled operand tiles start on 1 KB boundaries");

struct TcArgs {
  const uint16_t* q_cat;  // [B][128][576] bf16
  int* plan;              // read; the exact-recompute flags and context are written
  const uint8_t* pages;
  const int32_t* page_table;
  uint16_t* part_o;  // bf16 [128 heads][seg_cap segments][512]
  float* part_lse;
  int* err;
  int B, max_pages, num_pages;  // B: plan rows (virtual rows of the query layout)
  int seg_cap;                  // segments per head in part_o
  float scale_log2;
  QSpec qs;           // query layout: virtual row r reads page-table row r / qs.NG
  long long q_rows;   // flat rows of q_cat
};

// Bounded wait shared by all roles: gives up after WAIT_LIMIT_CYCLES (records
// MLA_ERR_TIMEOUT and raises the abort flag of this CTA and of its peer) or
// once an abort was raised.  The abort flag and the clock are checked every 8
// probes.
// error reports from hot loops, out of line
__device__ __noinline__ void report_error(int* err, int code, int info) { raise_error(err, code, info); }
// a row whose weights cannot be formed exactly here: the combine kernel recomputes it
__device__ __noinline__ void flag_row(int* fix, int b) { fix[b] = 1; }
// Query layout lookups, out of line (rare: at row changes, and only with several
// query tokens per row) so that the page loops' code stays small: the flat
// query row of a virtual row, its page-table row, a lane's causal shift.
__device__ __noinline__ long long qrow_of(const QSpec qs, int r) { return qs.qrow(r); }
__device__ __noinline__ int page_row_of(const QSpec qs, int r) { return r / qs.NG; }
__device__ __noinline__ int shift_of(const QSpec qs, int r, int v) { return qs.shift(r, v); }
__device__ __forceinline__ long long qrow_at(const QSpec& qs, int r) {
  return qs.NG == 1 ? (long long)r * qs.T * qs.Hr : qrow_of(qs, r);  // one virtual row per row: r * T * Hr
}
__device__ __forceinline__ int page_row_at(const QSpec& qs, int r) { return qs.NG == 1 ? r : page_row_of(qs, r); }

template <bool kCluster>
__device__ __forceinline__ bool probe_bar(uint64_t* bar, uint32_t parity) {
  return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
}
// the polling part, out of line: waits are many and usually end at the first
// probe, so the inlined part stays one instruction sequence per call site
template <bool kCluster>
__device__ __noinline__ bool wait_bar_slow(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err,
                                           int where) {
  const long long t0 = clock64();
  for (uint32_t k = 1;; ++k) {
    if (probe_bar<kCluster>(bar, parity)) return true;
    if ((k & 7) == 0) {
      if (*abort_flag) return false;
      if (clock64() - t0 > WAIT_LIMIT_CYCLES) {
        *abort_flag = 1;
        st_cluster_u32(mapa(smem_u32((const void*)abort_flag), cluster_ctarank() ^ 1u), 1u);
        report_error(err, MLA_ERR_TIMEOUT, where);
        return false;
      }
    }
  }
}
template <bool kCluster, class Smem>
__device__ __forceinline__ bool wait_bar(Smem& S, uint64_t* bar, uint32_t parity, int* err, int where) {
  if (probe_bar<kCluster>(bar, parity)) return true;
  return wait_bar_slow<kCluster>(bar, parity, &S.abort_flag, err, where);
}

// Per-lane TMEM passes over 128 O columns (whole warps call them): times f in
// place (a reference move, rare: out of line; the warp reconverges first, as
// the tcgen05 loads and stores are warp-aligned) ...
__device__ __noinline__ void scale_o_cols(uint32_t taddr, float f) {
  __syncwarp();
#pragma unroll 1
  for (int k16 = 0; k16 < 8; ++k16) {
    uint32_t o[16];
    const uint32_t col = taddr + 16 * k16;
    tmem_ld16(col, o);
    tmem_ld_wait();
#pragma unroll
    for (int k = 0; k < 16; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * f);
    tmem_st16(col, o);
  }
  tmem_st_wait();
}
// ... and times inv, rounded to bf16, into 128 values at dst (a segment's
// partial output; dst of lane l is row l).  Each 128-byte line of the rows is
// written by four lanes: the lanes of a group of four transpose their four
// rows' 32-byte chunks (two xor-shuffle stages), so a store instruction covers
// eight whole lines instead of 32 sectors of 32 lines.  Inlined: an
// out-of-line copy called from the segment-end branch returned wrong data.
__device__ __forceinline__ void store_o_cols(uint32_t taddr, uint16_t* dst, float inv) {
  const int lane = threadIdx.x & 31, j = lane & 3;
#pragma unroll 1
  for (int line = 0; line < 2; ++line) {  // 64 columns = 128 bytes of bf16
    uint32_t c[4][8];                      // c[k]: chunk k (16 values, 8 words) of a row of this group
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      uint32_t raw[32];
      tmem_ld32(taddr + 64 * line + 32 * hf, raw);
      tmem_ld_wait();
#pragma unroll
      for (int w = 0; w < 16; ++w)
        c[2 * hf + w / 8][w % 8] =
            pack_bf16x2(__uint_as_float(raw[2 * w]) * inv, __uint_as_float(raw[2 * w + 1]) * inv);
    }
    // 4 x 4 transpose of chunks across the group: afterwards c[s] of lane j is
    // chunk j of row s of the group
#pragma unroll
    for (int b = 2; b >= 1; b >>= 1) {
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        if (t & b) continue;  // t: the slot pair (t, t | b)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const bool hi = (j & b) != 0;
          const uint32_t send = hi ? c[t][e] : c[t | b][e];
          const uint32_t got = __shfl_xor_sync(0xffffffffu, send, b);
          if (hi) c[t][e] = got; else c[t | b][e] = got;
        }
      }
    }
    // row 4(lane/4) + s of the warp, chunk j of this line
#pragma unroll
    for (int s4 = 0; s4 < 4; ++s4) {
      uint16_t* p =
          reinterpret_cast<uint16_t*>(__shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(dst), (lane & ~3) | s4)) +
          64 * line + 16 * j;
      st_global_v8(reinterpret_cast<float*>(p), __uint_as_float(c[s4][0]), __uint_as_float(c[s4][1]),
                   __uint_as_float(c[s4][2]), __uint_as_float(c[s4][3]), __uint_as_float(c[s4][4]),
                   __uint_as_float(c[s4][5]), __uint_as_float(c[s4][6]), __uint_as_float(c[s4][7]));
    }
  }
}
// row of the tile cursor: tiles [start, end) belong to row b of length n
struct RowCursor {
  int b, start, end, n;
  __device__ __forceinline__ void init(const int* prefix, const int* seq_c, int row) {
    b = row;
    start = prefix[b];
    end = prefix[b + 1];
    n = seq_c[b];
  }
  // loads only when the tile moves to a later row
  __device__ __forceinline__ void advance(const int* prefix, const int* seq_c, int x) {
    while (x >= end) {
      ++b;
      start = end;
      end = prefix[b + 1];
      n = seq_c[b];
    }
  }
};

__device__ __forceinline__ float u2f(uint32_t v) { return __uint_as_float(v); }
// N (16 or 32) consecutive TMEM columns of this thread's lane
template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t* r) {
  static_assert(N == 16 || N == 32, "16 or 32 columns");
  if constexpr (N == 32) tmem_ld32(taddr, r); else tmem_ld16(taddr, r);
}
// two fp16 in one 32-bit word <-> two floats, in registers (low half = first
// value); the conversion saturates to the largest finite fp16 (+-65504)
__device__ __forceinline__ uint32_t f2_to_h2_sat(float lo, float hi) {
  uint32_t u;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(u) : "f"(hi), "f"(lo));
  return u;
}
__device__ __forceinline__ float2 h2_to_f2(uint32_t u) {
  __half2 h;
  memcpy(&h, &u, 4);
  return __half22float2(h);
}

// byte offset of 16-byte unit u (0..3, 8 tokens) of row r in a 64B-swizzled tile of 64-byte rows
// (the P half tiles, read by the tensor core, and the fp16 exchange tiles)
__device__ __forceinline__ uint32_t sw64(int r, int u) { return (uint32_t)(r * 64 + ((u ^ ((r >> 1) & 3)) << 4)); }

// ---- dequantization ("DeepSeek-V2-Lite MLA 吸收式 KV 缓存优化" §3.2 block
// quantizers): x = code * s (INT8), x = code * s + z (INT4), evaluated in fp32
// and rounded once to bf16 for the MMA.  Integer codes reach fp32 exactly by
// placing them in the low mantissa bits of 2^23 (a byte permute) and
// subtracting the offset; pairs of values go through the packed fp32 pipe
// (add/mul/fma.rn.f32x2), whose results equal the scalar ones (the code
// product with a bf16 scale is exact in fp32; INT4's fma rounds once).
__device__ __forceinline__ float bf16_to_f(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ uint64_t add_f2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t mul_f2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
__device__ __forceinline__ uint64_t fma_f2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
// two fp32 (one packed pair) rounded to a bf16x2 word (low half = first value)
__device__ __forceinline__ uint32_t f2_to_bf16x2(uint64_t v) {
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
  return pack_bf16x2(lo, hi);
}
// bytes k, k+1 of a word (already biased / masked into 0..255) as 2^23 + byte, packed
__device__ __forceinline__ uint64_t magic_pair(uint32_t w, int k) {
  return f2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7440u + (uint32_t)k)),
            __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7441u + (uint32_t)k)));
}
// bytes k, k+1 of a word of signed 8-bit codes times s2 = {s, s} -> bf16x2
__device__ __forceinline__ uint32_t deq_i8_pair(uint32_t biased, int k, uint64_t s2) {
  const uint64_t off = f2(-8388736.f, -8388736.f);  // -(2^23 + 128): the codes exactly
  return f2_to_bf16x2(mul_f2(add_f2(magic_pair(biased, k), off), s2));
}
// 8 signed 8-bit codes times s -> 8 bf16 (one 16-byte unit)
__device__ __forceinline__ uint4 deq_i8x8(uint32_t c0, uint32_t c1, float s) {
  const uint64_t s2 = f2(s, s);
  const uint32_t w0 = c0 ^ 0x80808080u, w1 = c1 ^ 0x80808080u;
  return make_uint4(deq_i8_pair(w0, 0, s2), deq_i8_pair(w0, 2, s2), deq_i8_pair(w1, 0, s2), deq_i8_pair(w1, 2, s2));
}
// 16 signed 8-bit codes (one 16-byte load) times s -> 16 bf16 (two 16-byte units)
__device__ __forceinline__ void deq_i8x16(uint4 c, float s, uint4& o0, uint4& o1) {
  const uint64_t s2 = f2(s, s);
  const uint32_t w0 = c.x ^ 0x80808080u, w1 = c.y ^ 0x80808080u, w2 = c.z ^ 0x80808080u, w3 = c.w ^ 0x80808080u;
  o0 = make_uint4(deq_i8_pair(w0, 0, s2), deq_i8_pair(w0, 2, s2), deq_i8_pair(w1, 0, s2), deq_i8_pair(w1, 2, s2));
  o1 = make_uint4(deq_i8_pair(w2, 0, s2), deq_i8_pair(w2, 2, s2), deq_i8_pair(w3, 0, s2), deq_i8_pair(w3, 2, s2));
}
// 8 unsigned 4-bit codes of one word (element 2i in the low nibble of byte i)
// as code * s + z -> 8 bf16 (one 16-byte unit)
__device__ __forceinline__ uint4 deq_u4x8(uint32_t w, uint64_t s2, uint64_t z2) {
  const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
  const uint64_t off = f2(-8388608.f, -8388608.f);  // -2^23
  uint32_t r[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint64_t m = f2(__uint_as_float(__byte_perm(lo, 0x4B000000u, 0x7440u + (uint32_t)i)),
                          __uint_as_float(__byte_perm(hi, 0x4B000000u, 0x7440u + (uint32_t)i)));
    r[i] = f2_to_bf16x2(fma_f2(add_f2(m, off), s2, z2));
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

// One staged page half (codes, scales, zeros of this CTA's dims) -> the bf16
// operand stage, by the 128 threads sid = 0..127 of the four PT warps.  Every
// thread owns fixed 16-byte code chunks:
//   INT8 latent: 64 tokens x 16 chunks of 16 codes; chunk k = sid + 128 i is
//     token k / 16, dims 16 (k % 16) .. (operand chunk (k % 16) / 4), scale
//     group (k % 16) / 2;
//   INT4 latent: 64 tokens x 8 chunks of 32 codes (one group each); chunk
//     k = sid + 128 i is token k / 8, group k % 8 (operand chunk (k % 8) / 2);
//   RoPE key (INT8 in both): token sid / 2, dims 16 (sid % 2) .., groups
//     4 rank + 2 (sid % 2) + {0, 1}.
// Tokens at or past nvalid are written as zeros.  A thread's latent rows share
// one swizzle (their tokens differ by multiples of 8).  The 8 lanes of a
// quarter warp (one phase of a 16-byte store) write 8 different 16-byte bank
// groups: the operand chunks are 8 KB apart (the same banks), so lanes of odd
// operand chunks store their two INT8 units in the other order, and INT4 lanes
// rotate their four units by the chunk index.  Out of line and rolled (with
// the next chunk's loads in flight): instruction fetch, not arithmetic, bounds
// this stage.
template <int FMT>
__device__ __noinline__ void dequant_page(const uint8_t* cd, uint8_t* kv, int nvalid, int sid, int rank) {
  using FT = FmtTraits<FMT>;
  constexpr bool kI8 = FMT == MLA_FMT_INT8;
  constexpr int NCH = kI8 ? 8 : 4, QN = kI8 ? 16 : 8, ROW = kI8 ? 256 : 128, TSTEP = 128 / QN;
  const int q = sid % QN, t0 = sid / QN, sw = t0 & 7;
  const int ci = kI8 ? q >> 2 : q >> 1, u0 = kI8 ? 2 * (q & 3) : 4 * (q & 1);
  const uint8_t* cp = cd + FT::C_OFF + t0 * ROW + 16 * q;
  const uint16_t* sp = reinterpret_cast<const uint16_t*>(cd + FT::CS_OFF) + t0 * 8 + (kI8 ? q >> 1 : q);
  const uint16_t* zp = reinterpret_cast<const uint16_t*>(cd + FT::ZS_OFF) + t0 * 8 + q;
  uint8_t* row = kv + ci * KV_CHUNK + t0 * 128;
  uint4 cn = *reinterpret_cast<const uint4*>(cp);
  uint16_t sn = sp[0], zn = kI8 ? 0 : zp[0];
#pragma unroll 1
  for (int i = 0; i < NCH; ++i) {
    const uint4 c = cn;
    const uint16_t sc = sn, zc = zn;
    const int nx = i + 1 < NCH ? i + 1 : i;  // the next chunk's loads go out now
    cn = *reinterpret_cast<const uint4*>(cp + nx * TSTEP * ROW);
    sn = sp[nx * TSTEP * 8];
    if constexpr (!kI8) zn = zp[nx * TSTEP * 8];
    const bool live = t0 + TSTEP * i < nvalid;
    uint8_t* r = row + i * TSTEP * 128;
    if constexpr (kI8) {
      const bool odd = ci & 1;  // store the second unit first
      uint4 o0 = make_uint4(0u, 0u, 0u, 0u), o1 = o0;
      if (live)
        deq_i8x16(odd ? make_uint4(c.z, c.w, c.x, c.y) : c, bf16_to_f(sc), o0, o1);
      *reinterpret_cast<uint4*>(r + (((u0 + (odd ? 1 : 0)) ^ sw) << 4)) = o0;
      *reinterpret_cast<uint4*>(r + (((u0 + (odd ? 0 : 1)) ^ sw) << 4)) = o1;
    } else {
      const float s1 = bf16_to_f(sc), z1 = bf16_to_f(zc);
      const uint64_t s2 = f2(s1, s1), z2 = f2(z1, z1);
      // the four words rotated by ci: store k writes unit (u0 + (k + ci) % 4)
      uint32_t w0 = c.x, w1 = c.y, w2 = c.z, w3 = c.w;
      if (ci & 1) { const uint32_t t = w0; w0 = w1; w1 = w2; w2 = w3; w3 = t; }
      if (ci & 2) { uint32_t t = w0; w0 = w2; w2 = t; t = w1; w1 = w3; w3 = t; }
      const uint32_t w[4] = {w0, w1, w2, w3};
#pragma unroll
      for (int k = 0; k < 4; ++k)
        *reinterpret_cast<uint4*>(r + (((u0 + ((k + ci) & 3)) ^ sw) << 4)) =
            live ? deq_u4x8(w[k], s2, z2) : make_uint4(0u, 0u, 0u, 0u);
    }
  }
  // RoPE key
  const int tp = sid >> 1, hh = sid & 1;
  const uint4 pw = *reinterpret_cast<const uint4*>(cd + FT::PE_OFF + tp * 32 + 16 * hh);
  const uint16_t* psc = reinterpret_cast<const uint16_t*>(cd + FT::PS_OFF) + tp * 8 + 4 * rank + 2 * hh;
  uint4 o0 = make_uint4(0u, 0u, 0u, 0u), o1 = o0;
  if (tp < nvalid) {
    o0 = deq_i8x8(pw.x, pw.y, bf16_to_f(psc[0]));  // dims 0..7: the first group's scale
    o1 = deq_i8x8(pw.z, pw.w, bf16_to_f(psc[1]));  // dims 8..15: the second's
  }
  uint8_t* pr = kv + KV_PE_OFF + tp * 64;
  const int psw = (tp >> 1) & 3;
  *reinterpret_cast<uint4*>(pr + (((2 * hh) ^ psw) << 4)) = o0;
  *reinterpret_cast<uint4*>(pr + (((2 * hh + 1) ^ psw) << 4)) = o1;
}

// The cache tensor maps: bf16 pages use m0 (latent, 128B-swizzled boxes of 64
// dims) and m1 (RoPE key, 64B-swizzled boxes of 32), and the query maps m2
// (q_lat: 128B-swizzled boxes of 64 dims x 128 heads) and m3 (q_pe:
// 64B-swizzled boxes of 32 dims x 64 heads); quantized pages use m0 (c codes),
// m1 (k_pe codes), m2 (c scales), m3 (INT4: c zeros, INT8: k_pe scales), m4
// (INT4: k_pe scales), and tm_q_pe (q_pe: 32 dims x 128 heads).
//
// Operand ring (bf16).  The producer streams ring "uses" in order: at the start
// of every segment two uses carry the segment's query (each: 128 heads x 128
// latent dims of this CTA's half, two 128B-swizzled tiles, plus 64 heads of its
// q_pe half), then one use per page.  Page i of segment k (both counted from 0
// within the worker) is use i + 2(k+1).  The S issuer of a segment's first page
// copies the query into TMEM (tcgen05.cp) and q_pe into qpe, then releases the
// two uses; no thread-issued global load is on the path of a segment change.
template <int FMT>
__global__ void __launch_bounds__(TC_THREADS, 1)
    attend_tc_kernel(const __grid_constant__ CUtensorMap tm_m0, const __grid_constant__ CUtensorMap tm_m1,
                     const __grid_constant__ CUtensorMap tm_m2, const __grid_constant__ CUtensorMap tm_m3,
                     const __grid_constant__ CUtensorMap tm_m4, const __grid_constant__ CUtensorMap tm_q_pe,
                     const TcArgs a) {
  using Smem = SmemTC<FMT>;
  using FT = FmtTraits<FMT>;
  constexpr bool kQuant = FMT != MLA_FMT_BF16;
  constexpr int KV_ST = Smem::KV_ST, CODE_ST = Smem::CODE_ST;
  extern __shared__ uint8_t smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
  const int worker = blockIdx.x >> 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < KV_ST; ++s) {
      mbar_init(&S.kv_full[s], kQuant ? 4 : 1);  // quantized: the 4 PT warps after dequantizing
      mbar_init(&S.kv_empty[s], 1);
    }
    for (int s = 0; s < CODE_ST; ++s) {
      mbar_init(&S.code_full[s], 1);
      mbar_init(&S.code_empty[s], 4);
    }
    mbar_init(&S.q_ready, 9);  // the 8 MT warps' q_lat + the q_pe copy
    mbar_init(&S.q_done, 1);
    mbar_init(&S.qpe_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&S.s_full[s], 1);
      mbar_init(&S.s_free[s], 12);  // every softmax warp
      mbar_init(&S.p_full[s], 8);  // each local MT warp once its P rows are written (expect_tx) + the peer's P rows
      mbar_init(&S.pv_done[s], 1);
      mbar_init(&S.pv_both[s], 2);   // this CTA's and the peer's P.V commits
      for (int q = 0; q < 4; ++q) {
        mbar_init(&S.x_full[s][q], 1);    // local expect_tx arrival + the peer's fp16 partial rows
        mbar_init(&S.x_empty[s][q], 2);   // one remote arrival per peer MT warp of the quadrant
        mbar_init(&S.pin_full[s][q], 3);  // expect_tx + the 2 local MT warps' messages + the peer's messages
      }
    }
    mbar_init(&S.o_free, 8);  // the MT warps' epilogues
    for (int q = 0; q < 4; ++q) {
      mbar_init(&S.mx_full[q], 3);   // expect_tx + the 2 local MT warps' maxima + the peer's maxima
      mbar_init(&S.mx_empty[q], 4);  // those maxima read by the 2 local and the 2 peer MT warps
    }
    for (int k = 0; k < 3; ++k) mbar_init(&S.mma_done[k], 1);
    S.abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  cluster_sync();  // the peer arrives on our barriers and writes our exchange buffers
  fence_after_sync();
  const uint32_t tmem = S.tmem_base;
  // everything above overlaps the end of the kernel before this one; the plan,
  // the query and the cache may come from it
  grid_dep_wait();
  grid_dep_launch();
  const int T = a.plan[0], W = a.plan[1], B = a.B;
  const int* prefix = a.plan + PLAN_HDR;
  const int* seq_c = a.plan + plan_off_seq(B);
  int* const fix = a.plan + plan_off_fix(B);
  // a plan may use fewer workers than this launch has CTA pairs: the rest idle
  const bool live = worker < W;
  const int row0 = live ? a.plan[plan_off_wrow(B) + worker] : 0;  // first row of this worker's range
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    // what the combine kernel reads to recompute a flagged row
    FixCtx* fx = reinterpret_cast<FixCtx*>(a.plan + PLAN_CTX);
    fx->pages = a.pages;
    fx->page_table = a.page_table;
    fx->q_cat = a.q_cat;
    fx->max_pages = a.max_pages;
    fx->num_pages = a.num_pages;
    fx->fmt = FMT;
    fx->scale_log2 = a.scale_log2;
    fx->qs = a.qs;
  }
  const int x0 = live ? (int)worker_begin(worker, T, W) : 0, x1 = live ? (int)worker_begin(worker + 1, T, W) : 0;
  const int ntiles = x1 - x0;

  // Roles of warps 0..3 (warp w runs on SM sub-partition w % 4; the pair's two
  // CTAs place them differently): role 0 producer, 1 P.V issuer, 2 / 3 S
  // issuers of even / odd pages.
  const int role = warp < 4 ? (warp ^ (int)(2 * rank)) : -1;
  if (ntiles > 0 && role == 0) {
    // ------------------------------------------------------------ TMA producer
    // The whole warp walks the pages; lane l holds the page id of tile
    // jbase + l of the current row (one gather per 32 tiles), lane 0 waits and
    // issues the copies.
    if (lane == 0) {
      prefetch_tmap(&tm_m0);
      prefetch_tmap(&tm_m1);
      if (kQuant) {
        if (FMT == MLA_FMT_INT4) prefetch_tmap(&tm_m4);
      }
      prefetch_tmap(&tm_m2);
      prefetch_tmap(&tm_m3);
    }
    const uint64_t pol = policy_evict_first();
    constexpr int RING = kQuant ? CODE_ST : KV_ST;  // slots the copies land in
    int issued = 0;  // ring uses whose copies were started (use k went to slot k % RING)
    RowCursor rc;
    rc.init(prefix, seq_c, row0);
    int page_row = -1, jbase = 0, page_reg = 0, seg = -1;
    for (int x = x0, i = 0; x < x1; ++x, ++i) {
      rc.advance(prefix, seq_c, x);
      const int j = x - rc.start;
      if (x == x0 || x == rc.start) ++seg;
      if (x == max(max(x0, rc.start), rc.end - Q_AHEAD) && rc.end < x1 && lane == 0) {
        // a few pages (this warp runs up to KV_ST pages ahead of the softmax)
        // before the end of a row whose segment is not this worker's last:
        // the next row's query is loaded at the row change; bring it into L2
        // with a high retention priority (each CTA of the pair half of it)
        RowCursor nx = rc;
        nx.advance(prefix, seq_c, rc.end);
        const long long qr = qrow_at(a.qs, nx.b) + 64 * rank;
        if (qr + 64 <= a.q_rows) prefetch_l2_bulk_hint(a.q_cat + qr * DK, 64 * DK * 2, policy_evict_last());
      }
      if (rc.b != page_row || j - jbase >= 32) {
        if (rc.b != page_row && rc.end < x1) {
          // entering a row whose segment is not this worker's last: warm L2
          // with the next row's page-table entries, which this warp needs at
          // the next segment change
          RowCursor nx = rc;
          nx.advance(prefix, seq_c, rc.end);
          const int32_t* pt = a.page_table + (size_t)page_row_at(a.qs, nx.b) * a.max_pages;
          const int nt = nx.end - nx.start;
          for (int k = 32 * lane; k < nt; k += 32 * 32) prefetch_l2_line(pt + k);
        }
        page_row = rc.b;
        jbase = j;
        page_reg = (j + lane < rc.end - rc.start)
                       ? a.page_table[(size_t)page_row_at(a.qs, rc.b) * a.max_pages + j + lane]
                       : 0;
      }
      int page = __shfl_sync(0xffffffffu, page_reg, j - jbase);
      int ok = 1;
      if constexpr (!kQuant) {
        if (lane == 0 && (x == x0 || x == rc.start)) {
          // the segment's query: two ring uses (q_lat dims [128h, 128h+128) of
          // this CTA's half and q_pe heads [64h, 64h+64) in use h)
          for (int h = 0; h < 2 && ok; ++h) {
            const int u = i + 2 * seg + h, st = u % KV_ST;
            ok = wait_bar<false>(S, &S.kv_empty[st], ((u / KV_ST) & 1) ^ 1, a.err, 1);
            if (ok) {
              mbar_arrive_expect_tx(&S.kv_full[st], 2 * QT_BYTES + QPE_BYTES / 2);
              const int qr = (int)qrow_at(a.qs, rc.b);  // flat query rows (past the end: zeros)
              for (int c = 0; c < 2; ++c)
                tma_load_3d(S.kv[st] + c * QT_BYTES, &tm_m2, HALF_C * rank + 128 * h + 64 * c, qr, 0, &S.kv_full[st]);
              tma_load_3d(S.kv[st] + 2 * QT_BYTES, &tm_m3, DC + PE_HALF * rank, qr + 64 * h, 0, &S.kv_full[st]);
              ++issued;
            }
          }
        }
      }
      if (lane == 0 && ok) {
        const int u = kQuant ? i : i + 2 * (seg + 1);  // ring use of this page
        const int st = u % RING;
        ok = wait_bar<false>(S, kQuant ? &S.code_empty[st] : &S.kv_empty[st], ((u / RING) & 1) ^ 1, a.err, 2);
        if (ok) {
          if (page < 0 || page >= a.num_pages) {
            report_error(a.err, MLA_ERR_BOUNDS, page);
            page = 0;
          }
          if constexpr (!kQuant) {
            mbar_arrive_expect_tx(&S.kv_full[st], KV_BYTES);
            for (int ci = 0; ci < 4; ++ci)
              tma_load_3d_hint(S.kv[st] + ci * KV_CHUNK, &tm_m0, HALF_C * rank + 64 * ci, 0, page, &S.kv_full[st],
                               pol);
            tma_load_3d_hint(S.kv[st] + KV_PE_OFF, &tm_m1, DC + PE_HALF * rank, 0, page, &S.kv_full[st], pol);
          } else {
            uint64_t* bar = &S.code_full[st];
            uint8_t* dst = S.code[st];
            mbar_arrive_expect_tx(bar, FT::CODE_BYTES);
            // c codes of this CTA's 256 latent dims (INT4: 128 bytes of them)
            tma_load_3d_hint(dst + FT::C_OFF, &tm_m0, (FMT == MLA_FMT_INT8 ? 256 : 128) * (int)rank, 0, page, bar,
                             pol);
            tma_load_3d_hint(dst + FT::PE_OFF, &tm_m1, PE_HALF * rank, 0, page, bar, pol);  // k_pe codes
            tma_load_3d_hint(dst + FT::CS_OFF, &tm_m2, 8 * rank, 0, page, bar, pol);        // c scales
            if constexpr (FMT == MLA_FMT_INT4) {
              tma_load_3d_hint(dst + FT::ZS_OFF, &tm_m3, 8 * rank, 0, page, bar, pol);  // c zeros
              tma_load_3d_hint(dst + FT::PS_OFF, &tm_m4, 0, 0, page, bar, pol);         // k_pe scales
            } else {
              tma_load_3d_hint(dst + FT::PS_OFF, &tm_m3, 0, 0, page, bar, pol);  // k_pe scales
            }
          }
          ++issued;
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
    }
    if (lane == 0 && S.abort_flag) {  // let copies in flight land before the CTA can exit
      for (int k = max(0, issued - RING); k < issued; ++k)
        (void)mbar_wait(kQuant ? &S.code_full[k % RING] : &S.kv_full[k % RING], (k / RING) & 1);
    }
  } else if (ntiles > 0 && (role == 2 || role == 3) && lane == 0) {
    // ------------------------------------------------------------ S issuers
    // warp 1: pages 0, 2, 4, ... of this worker; warp 2: pages 1, 3, 5, ...
    const int parity = role - 2;
    const uint32_t idesc_s = idesc_bf16_f32(128, TILE, false, false);
    const uint64_t qpe_desc = smem_desc(smem_u32(S.qpe), 16, 512, SWIZZLE_64B);
    int q_seen = 0;     // segments counted so far (the current one included)
    int q_have = 0;     // bf16: segments whose query this issuer has seen installed
    RowCursor rc;
    rc.init(prefix, seq_c, row0);
    for (int x = x0, i = 0; x < x1; ++x, ++i) {
      rc.advance(prefix, seq_c, x);
      const bool first = (x == x0) || (x == rc.start);
      if (first) ++q_seen;  // every issuer counts every segment
      if ((i & 1) != parity) continue;
      const int seg = q_seen - 1;
      const int u = kQuant ? i : i + 2 * (seg + 1);  // ring use of this page
      const int st = u % KV_ST, sb = i & 1;
      if constexpr (kQuant) {
        // the query of this page's segment is in place (TMEM half + smem q_pe)
        if (!wait_bar<false>(S, &S.q_ready, (uint32_t)seg & 1u, a.err, 3)) break;
      } else {
        if (first) {
          // install the segment's query: its two ring uses have landed, and the
          // previous segment's scores (the last reads of the old query) are done
          const int ua = u - 2, ub = u - 1;
          if (!wait_bar<false>(S, &S.kv_full[ua % KV_ST], (uint32_t)(ua / KV_ST) & 1u, a.err, 25)) break;
          if (!wait_bar<false>(S, &S.kv_full[ub % KV_ST], (uint32_t)(ub / KV_ST) & 1u, a.err, 26)) break;
          if (!wait_bar<false>(S, &S.s_free[sb], ((i >> 1) & 1) ^ 1, a.err, 5)) break;
          if (i > 0 && !wait_bar<false>(S, &S.s_full[(i - 1) & 1], (uint32_t)((i - 1) >> 1) & 1u, a.err, 27)) break;
          fence_after_sync();
          mbar_arrive_expect_tx(&S.qpe_full, QPE_BYTES);
#pragma unroll 1
          for (int h = 0; h < 2; ++h) {
            const uint32_t qa = smem_u32(S.kv[(u - 2 + h) % KV_ST]);
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)  // 16 dims per copy: TMEM columns of dims (2n, 2n+1)
                tmem_cp_128x256b(tmem + TM_Q + 64 * h + 32 * c + 8 * kk,
                                 smem_desc(qa + c * QT_BYTES + kk * 32, 16, 1024, SWIZZLE_128B));
            bulk_s2peer(mapa(smem_u32(S.qpe + h * (QPE_BYTES / 2)), rank), S.kv[(u - 2 + h) % KV_ST] + 2 * QT_BYTES,
                        QPE_BYTES / 2, mapa(smem_u32(&S.qpe_full), rank));
          }
          mma_commit(&S.q_done);
        }
        if (q_have < q_seen) {
          // the segment's query is in TMEM and smem (copied by whichever issuer
          // had its first page); that issuer then hands the two uses back
          if (!wait_bar<false>(S, &S.q_done, (uint32_t)seg & 1u, a.err, 28)) break;
          if (!wait_bar<false>(S, &S.qpe_full, (uint32_t)seg & 1u, a.err, 29)) break;
          q_have = q_seen;
          if (first) {
            mbar_arrive(&S.kv_empty[(u - 2) % KV_ST]);
            mbar_arrive(&S.kv_empty[(u - 1) % KV_ST]);
          }
        }
      }
      if (!wait_bar<false>(S, &S.kv_full[st], (uint32_t)(u / KV_ST) & 1u, a.err, 4)) break;
      if (!wait_bar<false>(S, &S.s_free[sb], ((i >> 1) & 1) ^ 1, a.err, 5)) break;
      fence_after_sync();
      const uint32_t kv_addr = smem_u32(S.kv[st]);
      const uint32_t d = tmem + TM_S + TILE * sb;
      const uint64_t bdesc = smem_desc(kv_addr, 16, 1024, SWIZZLE_128B);
      const uint64_t pdesc = smem_desc(kv_addr + KV_PE_OFF, 16, 512, SWIZZLE_64B);
#pragma unroll
      for (int ci = 0; ci < 4; ++ci)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts(d, tmem + TM_Q + ci * 32 + kk * 8, bdesc + (uint64_t)((ci * KV_CHUNK + kk * 32) >> 4), idesc_s,
                 (ci | kk) != 0 ? 1u : 0u);
#pragma unroll
      for (int kk = 0; kk < 2; ++kk)
        mma_ss(d, qpe_desc + (uint64_t)((kk * 32) >> 4), pdesc + (uint64_t)((kk * 32) >> 4), idesc_s, 1u);
      mma_commit(&S.s_full[sb]);
    }
    mma_commit(&S.mma_done[parity]);
    (void)mbar_wait(&S.mma_done[parity], 0);  // every issued MMA has finished
  } else if (ntiles > 0 && role == 1 && lane == 0) {
    // ------------------------------------------------------------ P.V issuer
    const uint32_t idesc_pv = idesc_bf16_f32(128, HALF_C, false, true);
    int segments = 0;
    RowCursor rc;
    rc.init(prefix, seq_c, row0);
    for (int x = x0, i = 0; x < x1; ++x, ++i) {
      rc.advance(prefix, seq_c, x);
      const bool first = (x == x0) || (x == rc.start);
      const int st = (kQuant ? i : i + 2 * (segments + (first ? 1 : 0))) % KV_ST, pb = i & 1;  // ring use of page i
      if (!wait_bar<false>(S, &S.p_full[pb], (i >> 1) & 1, a.err, 6)) break;
      // the first page of a segment overwrites O: wait for the previous
      // segment's epilogue to have read it
      if (first) {
        if (segments > 0 && !wait_bar<false>(S, &S.o_free, (segments - 1) & 1, a.err, 7)) break;
        ++segments;
      }
      fence_after_sync();
      fence_proxy_async_smem();  // P written or rescaled by this CTA's threads -> tensor core
      const uint64_t vdesc = smem_desc(smem_u32(S.kv[st]), KV_CHUNK, 1024, SWIZZLE_128B);
#pragma unroll
      for (int kk = 0; kk < TILE / 16; ++kk) {
        // tokens 16kk..16kk+15: P tile kk (computed by CTA kk / 2)
        const uint64_t adesc = smem_desc(smem_u32(S.p[pb][kk]), 16, 256, SWIZZLE_32B);
        mma_ss(tmem + TM_O, adesc, vdesc + (uint64_t)((kk * 16 * 128) >> 4), idesc_pv, (first && kk == 0) ? 0u : 1u);
      }
      mma_commit(&S.pv_done[pb]);
      mma_commit_mc(&S.pv_both[pb], (uint16_t)0x3);
      mma_commit(&S.kv_empty[st]);
    }
    mma_commit(&S.mma_done[2]);
    (void)mbar_wait(&S.mma_done[2], 0);
  } else if (ntiles > 0 && warp >= SOFT_WARP0) {
    // ------------------------------------------------------------ softmax warps
    const int q4 = warp & 3;                  // TMEM lane quadrant
    const int sub = (warp - SOFT_WARP0) >> 2;  // 0, 1: MT slice; 2: PT
    const int row = q4 * 32 + lane;           // head = TMEM lane
    const int stid = threadIdx.x - 32 * SOFT_WARP0;  // 0..255
    const uint32_t t_row = tmem + ((uint32_t)(q4 * 32) << 16);
    const float c = a.scale_log2;  // > 0
    RowCursor rc;
    rc.init(prefix, seq_c, row0);

    // the query of row b into place: the q_lat half into TMEM (each thread its
    // 2*QCOLS latent dims), the q_pe half into shared memory by one TMA copy
    auto load_query = [&](int b) {
      // flat query row of this lane (rows past the end of q_cat read as zeros)
      const long long qr = qrow_at(a.qs, b) + row;
      const bool have = qr < a.q_rows;
      const uint16_t* qrow = a.q_cat + (have ? qr : 0) * DK;
      const uint4* qc = reinterpret_cast<const uint4*>(qrow + HALF_C * rank + 2 * QCOLS * sub);
      // every global read is issued before the first TMEM store (one round trip)
      uint32_t v[QCOLS];
#pragma unroll
      for (int k = 0; k < QCOLS / 4; ++k) {
        const uint4 u = have ? qc[k] : make_uint4(0u, 0u, 0u, 0u);
        v[4 * k] = u.x; v[4 * k + 1] = u.y; v[4 * k + 2] = u.z; v[4 * k + 3] = u.w;
      }
#pragma unroll
      for (int k32 = 0; k32 < QCOLS / 32; ++k32) tmem_st32(t_row + TM_Q + QCOLS * sub + 32 * k32, v + 32 * k32);
      tmem_st_wait();
      fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.q_ready);
      if (stid == 0) {
        mbar_arrive_expect_tx(&S.q_ready, QPE_BYTES);
        tma_load_3d(S.qpe, &tm_q_pe, DC + PE_HALF * rank, (int)qrow_at(a.qs, b), 0, &S.q_ready);
      }
    };
    // The pair splits every page by token half: CTA r runs the softmax of all
    // 128 heads over tokens [32r, 32r+32) ("my" tokens).  In each lane quadrant
    // the warps with sub 0, 1 ("MT") own 16 of my tokens each and keep O (128
    // columns each) and the query; the warp with sub 2 ("PT") ships the peer's
    // 32 tokens' partial scores and, for quantized pools, dequantizes the next
    // page.
    const bool mt = sub < 2;
    const int ms = sub & 1;                   // MT: slice index within the token half
    auto scale_o = [&](float f) { scale_o_cols(t_row + TM_O + 128 * ms, f); };
    auto store_o = [&](int seg, float inv) {
      store_o_cols(t_row + TM_O + 128 * ms, a.part_o + ((size_t)row * a.seg_cap + seg) * DC + HALF_C * rank + 128 * ms,
                   inv);
    };

    bool failed = false;
    if (kQuant && mt) load_query(rc.b);  // bf16: the S issuers install each segment's query
    if (mt) {
      // ---------------------------------------------------------- MT warps
      // Exchange with the peer, per lane quadrant q4 and without group-wide
      // barriers: this warp ships its own P rows (1 KB, counted on the peer's
      // p_full[sb]) and message (128 B, on the peer's pin_full[sb][q4]) by bulk
      // copies.  p_full[sb] completes once all 8 local MT warps wrote their P
      // rows and the peer's 8 KB arrived: the P.V of the page needs nothing
      // else.  The two local MT warps of a quadrant also arrive on their own
      // pin_full after writing their messages, so a check sees all four slices
      // of its heads.
      const bool qlead = ms == 0 && lane == 0;  // arms this quadrant's barriers each page
      const int slot = 2 * (int)rank + ms;      // this warp's slice among the four of a page
      const uint32_t peer_xempty = mapa(smem_u32(&S.x_empty[0][q4]), peer);
      const uint32_t peer_pin = mapa(smem_u32(&S.pin_full[0][q4]), peer);
      const uint32_t peer_pfull = mapa(smem_u32(&S.p_full[0]), peer);
      const uint32_t peer_mxf = mapa(smem_u32(&S.mx_full[q4]), peer);
      const uint32_t peer_mxe = mapa(smem_u32(&S.mx_empty[q4]), peer);
      const uint32_t peer_p = mapa(smem_u32(&S.p[0][slot][0]), peer) + PG_Q * q4;
      const uint32_t peer_msg = mapa(smem_u32(&S.msgs[0][slot][0]), peer) + SL_Q * q4;
      constexpr uint32_t MX_Q = 32 * 2;  // one MT warp's first-page maxima (bf16)
      const uint32_t peer_mx = mapa(smem_u32(&S.mxs[slot][0]), peer) + MX_Q * q4;
      constexpr uint32_t BAR_SB = 4 * 8;                    // bytes between the page parities' quadrant barriers
      constexpr uint32_t P_SB = 4 * PG_BYTES, M_SB = 4 * 128 * 4;  // bytes between pages of the P / message rings
      const int tok0 = HALF_T * (int)rank + TPW * ms;  // first page token of this thread's slice
      // offset of 16-byte unit k (8 tokens) of this lane's row in a P tile
      const uint32_t prow = (uint32_t)row * 32;
      auto punit = [&](int k) -> uint32_t { return prow + ((uint32_t)(k ^ ((row >> 2) & 1)) << 4); };
      // softmax state of this head (lane), log2 domain:
      //  m_ref       reference of the P written from now on
      //  l           sum of this slice's p over the segment so far, in m_ref
      //  alpha_prev  factor of the reference move made at the last check (1 if none)
      float m_ref = -INFINITY, l = 0.f, alpha_prev = 1.f;
      int fcnt = 0;  // segment starts seen (phases of mx_full, mx_empty)
      // tokens at the end of the row's view that this lane's query does not see
      // (several query tokens per row: causal; padding lanes see nothing).  Such
      // a lane can have a whole segment masked: its reference stays -inf, its p
      // are 0, and its segment is stored as O = 0, LSE = -inf.
      int shift = 0;
      // check of page j, at the end of page j+1 (so it waits for nothing in
      // the common case): the four slice messages of page j have arrived.  If
      // page j's maximum exceeded its reference by more than RESCALE_LOG2 the
      // reference moves: the P of pages <= j+1 is already in the old one, so O
      // is rescaled once page j+1's P.V has completed (before page j+2's, which
      // needs this warp's next P), and l with it.  At a segment end the output
      // is written.  ref_j: the reference in force after the check of page j-1,
      // in which O and l hold page j (its P may have been written in the one
      // before and rescaled by that check).
      auto check = [&](int j, bool j_last, int seg, float ref_j) -> bool {
        const int jb = j & 1;
        bool ok = wait_bar<true>(S, &S.pin_full[jb][q4], (uint32_t)(j >> 1) & 1u, a.err, 20);
        __syncwarp();
        const int jm = j & 3;
        const float m0 = S.msgs[jm][0][row], m1 = S.msgs[jm][1][row], m2 = S.msgs[jm][2][row],
                    m3 = S.msgs[jm][3][row];
        if (!j_last) {
          // page j's maximum over all four slices against the reference it used
          const float m_comb = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
          float alpha = 1.f;
          if (m_comb > ref_j + RESCALE_LOG2) {
            const float m_new = fmaxf(m_comb, m_ref);
            alpha = ex2(m_ref - m_new);
            l *= alpha;  // the sums of pages <= j+1
            m_ref = m_new;  // pages from j+2 on
          }
          alpha_prev = alpha;
          if (__any_sync(0xffffffffu, alpha != 1.f)) {
            if (!wait_bar<false>(S, &S.pv_done[(j + 1) & 1], ((j + 1) >> 1) & 1, a.err, 21)) ok = false;
            __syncwarp();
            fence_after_sync();
            scale_o(alpha);
            fence_before_sync();
          }
        } else {
          // the four slices' sums were sent before the check of page j-1, so
          // they miss that check's move; O has it.  L is the sum in ref_j, the
          // reference after that move, and the log-sum-exp is taken in it too
          // (with Lm it would overstate the segment by the move whenever a
          // segment's second-to-last page moved the reference)
          const float Lm = (m0 + m1) + (m2 + m3);
          const float L = alpha_prev * Lm;
          alpha_prev = 1.f;
          if (!wait_bar<false>(S, &S.pv_done[jb], (uint32_t)(j >> 1) & 1u, a.err, 22)) ok = false;
          __syncwarp();
          fence_after_sync();
          store_o(seg, L > 0.f ? 1.f / L : 0.f);  // a segment this lane sees nothing of: O = 0
          if (rank == 0 && ms == 0) a.part_lse[(size_t)seg * 128 + row] = (ref_j + log2f(L)) * 0.69314718055994531f;
          fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(&S.o_free);
        }
        return ok;
      };
      int pend_i = -1, pend_seg = 0;
      bool pend_last = false;
      float pend_ref = 0.f;
      // one pass more than there are pages: the last one only checks the last
      // page (a single call site keeps the loop's code compact)
      for (int x = x0, i = 0; x <= x1; ++x, ++i) {
        bool last = false;
        if (x < x1) {
        rc.advance(prefix, seq_c, x);
        const bool first = (x == x0) || (x == rc.start);
        last = (x + 1 == x1) || (x + 1 == rc.end);
        if (first) shift = a.qs.G > 1 ? shift_of(a.qs, rc.b, row) : 0;
        // tokens of this page this lane's query sees (may be <= 0)
        const int nvalid = min(TILE, rc.n - shift - TILE * (x - rc.start));
        const int sb = i & 1;
        const uint32_t ph = (uint32_t)(i >> 1) & 1u;

        if (qlead) {
          mbar_arrive_expect_tx(&S.x_full[sb][q4], X_Q);     // the peer's partials of my tokens, these rows
          mbar_arrive_expect_tx(&S.pin_full[sb][q4], PIN_Q);  // the peer's messages
          if (first) mbar_arrive_expect_tx(&S.mx_full[q4], 2 * MX_Q);  // the peer's first-page maxima
        }
        // ---- this CTA's partial scores of my tokens; the S buffer is released
        if (!wait_bar<false>(S, &S.s_full[sb], ph, a.err, 9)) break;
        __syncwarp();
        fence_after_sync();
        uint32_t own[TPW];
        tmem_ld_cols<TPW>(t_row + TM_S + TILE * sb + tok0, own);
        tmem_ld_wait();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.s_free[sb]);

        // ---- add the peer's partial (fp16, log2 units) of my tokens
        if (!wait_bar<true>(S, &S.x_full[sb][q4], ph, a.err, 11)) break;
        __syncwarp();
        float s[TPW];
        const uint8_t* xi = S.xin[sb];
#pragma unroll
        for (int k = 0; k < TPW / 8; ++k) {
          const uint4 v = *reinterpret_cast<const uint4*>(xi + sw64(row, (TPW / 8) * ms + k));
          const float2 f0 = h2_to_f2(v.x), f1 = h2_to_f2(v.y), f2 = h2_to_f2(v.z), f3 = h2_to_f2(v.w);
          s[8 * k + 0] = fmaf(u2f(own[8 * k + 0]), c, f0.x);
          s[8 * k + 1] = fmaf(u2f(own[8 * k + 1]), c, f0.y);
          s[8 * k + 2] = fmaf(u2f(own[8 * k + 2]), c, f1.x);
          s[8 * k + 3] = fmaf(u2f(own[8 * k + 3]), c, f1.y);
          s[8 * k + 4] = fmaf(u2f(own[8 * k + 4]), c, f2.x);
          s[8 * k + 5] = fmaf(u2f(own[8 * k + 5]), c, f2.y);
          s[8 * k + 6] = fmaf(u2f(own[8 * k + 6]), c, f3.x);
          s[8 * k + 7] = fmaf(u2f(own[8 * k + 7]), c, f3.y);
        }
        if (nvalid < TILE) {
#pragma unroll
          for (int k = 0; k < TPW; ++k)
            if (tok0 + k >= nvalid) s[k] = -INFINITY;
        }
        float mraw = s[0];
#pragma unroll
        for (int k = 1; k < TPW; ++k) mraw = fmaxf(mraw, s[k]);

        // ---- the reference of this page's P
        if (first) {
          // segment start: the exact row maximum over the page's four slices
          const uint32_t fph = (uint32_t)(fcnt++) & 1u;
          if (!wait_bar<true>(S, &S.mx_empty[q4], fph ^ 1u, a.err, 18)) break;  // the last ones were read
          __syncwarp();
          {
            const __nv_bfloat16 mb = __float2bfloat16_rn(mraw);
            S.mxs[slot][row] = *reinterpret_cast<const uint16_t*>(&mb);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            bulk_s2peer(peer_mx, &S.mxs[slot][32 * q4], MX_Q, peer_mxf);
            mbar_arrive(&S.mx_full[q4]);
          }
          if (!wait_bar<true>(S, &S.mx_full[q4], fph, a.err, 19)) break;
          __syncwarp();
          m_ref = fmaxf(fmaxf(bf16_to_f(S.mxs[0][row]), bf16_to_f(S.mxs[1][row])),
                        fmaxf(bf16_to_f(S.mxs[2][row]), bf16_to_f(S.mxs[3][row])));
          __syncwarp();
          if (lane == 0) {  // both CTAs may write their maxima of the next segment start
            mbar_arrive(&S.mx_empty[q4]);
            mbar_arrive_remote_relaxed(peer_mxe);
          }
          l = 0.f;
        }
        if (mraw - m_ref > RANGE_LOG2) flag_row(fix, rc.b);
        // p = 2^(s - m_ref), rounded to bf16 for the MMA (exponent capped at
        // RANGE_LOG2: beyond it the row was flagged above for the exact recompute)
        uint32_t pk[TPW / 2];
        float sum0 = 0.f, sum1 = 0.f;
        const float mr = fmaxf(m_ref, -3.0e38f);  // m_ref = -inf only when every s is -inf (p = 0)
#pragma unroll
        for (int k = 0; k < TPW / 2; ++k) {
          const float p0 = ex2(fminf(s[2 * k] - mr, RANGE_LOG2));
          const float p1 = ex2(fminf(s[2 * k + 1] - mr, RANGE_LOG2));
          sum0 += p0;
          sum1 += p1;
          pk[k] = pack_bf16x2(p0, p1);
        }
        l += sum0 + sum1;
        // P tile sb is free once the P.V of page i-2 has completed in both CTAs
        if (!wait_bar<true>(S, &S.pv_both[sb], ph ^ 1u, a.err, 13)) break;
        __syncwarp();
        uint8_t* pm = S.p[sb][slot];
#pragma unroll
        for (int k = 0; k < 2; ++k)
          *reinterpret_cast<uint4*>(pm + punit(k)) = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
        // message: this slice's maximum, or its sum at a segment's last page
        S.msgs[i & 3][slot][row] = last ? l : mraw;
        // every value read from the exchange buffer has been used by the store
        // above (mraw depends on all of them), so the peer may refill it
        __syncwarp();
        if (lane == 0) mbar_arrive_remote_relaxed(peer_xempty + BAR_SB * sb);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          bulk_s2peer(peer_p + P_SB * sb, pm + PG_Q * q4, PG_Q, peer_pfull + 8u * sb);
          bulk_s2peer(peer_msg + M_SB * (i & 3), &S.msgs[i & 3][slot][32 * q4], SL_Q, peer_pin + BAR_SB * sb);
          mbar_arrive_expect_tx(&S.p_full[sb], PG_Q);  // our P rows; the peer's counterpart rows
          mbar_arrive(&S.pin_full[sb][q4]);            // our message, for our partner's check
        }
        // the next page starts a new segment: every S of this one has completed
        // (this thread waited for each), so the next query may replace this one
        if (kQuant && last && x + 1 < x1) {
          RowCursor nx = rc;
          nx.advance(prefix, seq_c, x + 1);
          load_query(nx.b);
        }
        }
        if (pend_i >= 0 && !check(pend_i, pend_last, pend_seg, pend_ref)) break;
        if (x == x1) break;
        pend_i = i;
        pend_last = last;
        pend_seg = worker + rc.b;
        pend_ref = m_ref;
      }
    } else {
      // ---------------------------------------------------------- PT warps
      constexpr int NSEND = 128;                       // PT threads
      const int sid = q4 * 32 + lane;                  // 0..NSEND-1
      // this warp ships its quadrant's rows (2 KB) to the peer's x_full[sb][q4]
      const uint32_t peer_xin = mapa(smem_u32(S.xin[0]), peer) + X_Q * q4;
      const uint32_t peer_xfull = mapa(smem_u32(&S.x_full[0][q4]), peer);
      constexpr uint32_t BAR_SB = 4 * 8;  // bytes between the page parities' quadrant barriers
      const int tok0 = HALF_T * (int)peer;             // the peer's token half
      // quantized formats: page j's staged codes -> bf16 operand stage j % KV_ST
      // (rows at or past nvalid are written as zeros), then release both
      auto dequant = [&](int j, int nvalid) -> bool {
        const int st = j % KV_ST, cs = j % CODE_ST;
        bool ok = wait_bar<false>(S, &S.code_full[cs], (uint32_t)(j / CODE_ST) & 1u, a.err, 23);
        // the P.V that last read this operand stage has completed
        if (!wait_bar<false>(S, &S.kv_empty[st], ((uint32_t)(j / KV_ST) & 1u) ^ 1u, a.err, 24)) ok = false;
        __syncwarp();
        if constexpr (kQuant) dequant_page<FMT>(S.code[cs], S.kv[st], nvalid, sid, (int)rank);
        fence_proxy_async_smem();  // generic writes -> the tensor core's reads
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&S.kv_full[st]);
          mbar_arrive(&S.code_empty[cs]);
        }
        return ok;
      };
      RowCursor rn;  // row of the page being dequantized
      if constexpr (kQuant) {
        // two pages ahead of the S MMAs: pages 0 and 1 now, page i+2 at page i
        rn.init(prefix, seq_c, row0);
        for (int x = x0; x < min(x0 + 2, x1) && !failed; ++x) {
          rn.advance(prefix, seq_c, x);
          if (!dequant(x - x0, min(TILE, rn.n - TILE * (x - rn.start)))) failed = true;
        }
      }
      int pseg = -1;  // segment of the page (bf16: two ring uses of query each)
      for (int x = x0, i = 0; x < x1; ++x, ++i) {
        rc.advance(prefix, seq_c, x);
        if (x == x0 || x == rc.start) ++pseg;
        const int nvalid = min(TILE, rc.n - TILE * (x - rc.start));
        const int st = (kQuant ? i : i + 2 * (pseg + 1)) % KV_ST, sb = i & 1;
        const uint32_t ph = (uint32_t)(i >> 1) & 1u;

        if (!wait_bar<false>(S, &S.s_full[sb], ph, a.err, 15)) break;
        __syncwarp();
        fence_after_sync();
        uint32_t v[HALF_T];
        tmem_ld32(t_row + TM_S + TILE * sb + tok0, v);
        tmem_ld_wait();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.s_free[sb]);
        if (!kQuant && nvalid < TILE) {
          // page past the end of its sequence: zero the unused value rows so that
          // P = 0 never meets stale (possibly non-finite) cache contents
          // (quantized pages: the dequantization writes those rows as zeros)
          const int units = (TILE - nvalid) * 4 * 8;  // 16-byte units in 4 chunks of 128-byte rows
          for (int idx = sid; idx < units; idx += NSEND) {
            const int r = nvalid + idx / 32, ci = (idx % 32) / 8, u = idx % 8;
            *reinterpret_cast<uint4*>(S.kv[st] + ci * KV_CHUNK + r * 128 + u * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();
        }
        uint32_t h[HALF_T / 2];
#pragma unroll
        for (int k = 0; k < HALF_T / 2; ++k) h[k] = f2_to_h2_sat(u2f(v[2 * k]) * c, u2f(v[2 * k + 1]) * c);
        // the peer has consumed what we sent into its buffer two pages ago (so
        // the copy that read xout[sb] then has completed too); with a single
        // staging tile, also last page's
        if (!wait_bar<true>(S, &S.x_empty[sb][q4], ph ^ 1u, a.err, 16)) break;
        if (Smem::XOUT_N == 1 && i > 0 &&
            !wait_bar<true>(S, &S.x_empty[sb ^ 1][q4], (uint32_t)((i - 1) >> 1) & 1u, a.err, 17))
          break;
        __syncwarp();
        uint8_t* xo = S.xout[sb % Smem::XOUT_N];
#pragma unroll
        for (int k = 0; k < HALF_T / 8; ++k)
          *reinterpret_cast<uint4*>(xo + sw64(row, k)) = make_uint4(h[4 * k], h[4 * k + 1], h[4 * k + 2], h[4 * k + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) bulk_s2peer(peer_xin + sb * X_BYTES, xo + X_Q * q4, X_Q, peer_xfull + BAR_SB * sb);
        // after the copy is on its way (the peer waits for it, not for this): the
        // exactness check of the shipped half scores of the page's valid tokens
        {
          const int lim = nvalid - tok0;  // valid tokens of the shipped half
          float amax = 0.f;
#pragma unroll
          for (int k = 0; k < HALF_T; ++k)
            if (k < lim) amax = fmaxf(amax, fabsf(u2f(v[k])));
          if (amax * c > EXCH_LOG2) flag_row(fix, rc.b);
        }
        if constexpr (kQuant) {
          // page i+2's operands (its stage was last read by page i+2-KV_ST's P.V)
          if (x + 2 < x1) {
            rn.advance(prefix, seq_c, x + 2);
            if (!dequant(i + 2, min(TILE, rn.n - TILE * (x + 2 - rn.start)))) break;
          }
        }
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  fence_before_sync();
  __syncthreads();
  cluster_sync();  // the peer no longer touches our shared memory
  if (warp == 1) {
    fence_after_sync();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Self-test of the failure path of the waits above: a CTA pair in which CTA 0
// waits on a barrier that nothing completes.  Its wait gives up after
// WAIT_LIMIT_CYCLES, records MLA_ERR_TIMEOUT (detail 1) and raises the abort
// flags of both CTAs; CTA 1 starts its own wait a quarter of the limit later
// and leaves it through the abort flag.  Every wait is bounded: the kernel
// returns and nothing faults.
struct SelftestSmem {
  uint64_t bar;
  int abort_flag;
};
__global__ void __launch_bounds__(32, 1) wait_selftest_kernel(int* err) {
  __shared__ SelftestSmem S;
  const uint32_t rank = cluster_ctarank();
  if (threadIdx.x == 0) {
    mbar_init(&S.bar, 1);
    S.abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  cluster_sync();  // both flags are initialised before either CTA can raise the other's
  if (threadIdx.x == 0) {
    if (rank == 1) {
      const long long t0 = clock64();
      while (clock64() - t0 < WAIT_LIMIT_CYCLES / 4 && !*reinterpret_cast<volatile int*>(&S.abort_flag)) {
      }
    }
    (void)wait_bar<true>(S, &S.bar, 0, err, 1 + (int)rank);
  }
  __syncwarp();
  cluster_sync();  // neither CTA leaves while the other may still write its flag
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
template <int FMT>
constexpr size_t smem_bytes() { return sizeof(SmemTC<FMT>) + 1024; }

std::mutex g_tc_mu;
int g_tc_workers[64] = {};

cudaLaunchConfig_t launch_config(int workers, cudaStream_t s, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * workers);
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = smem_bytes<MLA_FMT_BF16>();
  cfg.stream = s;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see grid_dep_wait in the kernel
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

}  // namespace

cudaError_t launch_wait_selftest(int* err, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(32);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, wait_selftest_kernel, err);
}

// persistent workers (CTA pairs) that fit on the device at once
int attend_tc_workers(int num_sms) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms / 2;
  std::lock_guard<std::mutex> lk(g_tc_mu);
  if (g_tc_workers[dev] == 0) {
    int clusters = 0;
    if (cudaFuncSetAttribute(attend_tc_kernel<MLA_FMT_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem_bytes<MLA_FMT_BF16>()) == cudaSuccess) {
      cudaLaunchAttribute attr[2];
      cudaLaunchConfig_t cfg = launch_config(num_sms / 2, nullptr, attr);
      if (cudaOccupancyMaxActiveClusters(&clusters, attend_tc_kernel<MLA_FMT_BF16>, &cfg) != cudaSuccess) clusters = 0;
    }
    (void)cudaGetLastError();
    g_tc_workers[dev] = clusters > 0 ? std::min(clusters, num_sms / 2) : num_sms / 2;
  }
  return g_tc_workers[dev];
}

cudaError_t launch_attend_tc(const void* q_cat, const QSpec& qs, int fmt, int num_pages, const void* pages,
                             const int32_t* page_table, int max_pages, int Bv, float scale, int* plan,
                             int workers, int seg_cap, uint16_t* part_o, float* part_lse, int* err, cudaStream_t s) {
  if (qs.G * qs.Hr != 128 || qs.T < 1 || qs.NG != (qs.T + qs.G - 1) / qs.G || workers < 1) return cudaErrorNotSupported;
  if (fmt != MLA_FMT_BF16 && fmt != MLA_FMT_INT8 && fmt != MLA_FMT_INT4) return cudaErrorNotSupported;
  if (!(scale > 0.f)) return cudaErrorInvalidValue;  // the row max is taken before scaling
  const long long q_rows = (long long)(Bv / qs.NG) * qs.T * qs.Hr;
  if (q_rows > 2147483647LL - 256) return cudaErrorNotSupported;  // query rows are TMA coordinates
  CUtensorMap m[5], tq_pe;
  const uint64_t row = (uint64_t)DK * 2;  // 1,152 bytes per bf16 token slot / query row
  const uint8_t* pg = static_cast<const uint8_t*>(pages);
  const uint64_t P = (uint64_t)num_pages;
  const uint64_t QR = (uint64_t)q_rows;
  const CUtensorMapDataType U8 = CU_TENSOR_MAP_DATA_TYPE_UINT8, BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const CUtensorMapSwizzle NS = CU_TENSOR_MAP_SWIZZLE_NONE;
  // the query: flat rows of 576 (a virtual row's 128 virtual heads are 128
  // consecutive rows from qs.qrow(r)); rows past the end read as zeros
  bool ok = encode_3d(&tq_pe, q_cat, DK, QR, 1, row, row * QR, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B);
  if (fmt == MLA_FMT_BF16) {
    ok = ok && encode_3d(&m[0], pg, DK, PAGE, P, row, PAGE_BYTES_BF16, 64, TILE, CU_TENSOR_MAP_SWIZZLE_128B) &&
         encode_3d(&m[1], pg, DK, PAGE, P, row, PAGE_BYTES_BF16, 32, TILE, CU_TENSOR_MAP_SWIZZLE_64B) &&
         encode_3d(&m[2], q_cat, DK, QR, 1, row, row * QR, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) &&
         encode_3d(&m[3], q_cat, DK, QR, 1, row, row * QR, 32, 64, CU_TENSOR_MAP_SWIZZLE_64B);
    m[4] = m[0];
  } else if (fmt == MLA_FMT_INT8) {
    const uint64_t PB = PAGE_BYTES_INT8;  // sections at 0, 32768, 36864, 38912
    ok = ok && encode_3d(&m[0], pg, DC, PAGE, P, DC, PB, 256, TILE, NS, U8) &&
         encode_3d(&m[1], pg + 32768, DR, PAGE, P, DR, PB, 32, TILE, NS, U8) &&
         encode_3d(&m[2], pg + 36864, DC / 32, PAGE, P, (DC / 32) * 2, PB, 8, TILE, NS, BF) &&
         encode_3d(&m[3], pg + 38912, DR / 8, PAGE, P, (DR / 8) * 2, PB, 8, TILE, NS, BF);
    m[4] = m[0];
  } else {
    const uint64_t PB = PAGE_BYTES_INT4;  // sections at 0, 16384, 20480, 22528, 24576
    ok = ok && encode_3d(&m[0], pg, DC / 2, PAGE, P, DC / 2, PB, 128, TILE, NS, U8) &&
         encode_3d(&m[1], pg + 16384, DR, PAGE, P, DR, PB, 32, TILE, NS, U8) &&
         encode_3d(&m[2], pg + 20480, DC / 32, PAGE, P, (DC / 32) * 2, PB, 8, TILE, NS, BF) &&
         encode_3d(&m[3], pg + 22528, DC / 32, PAGE, P, (DC / 32) * 2, PB, 8, TILE, NS, BF) &&
         encode_3d(&m[4], pg + 24576, DR / 8, PAGE, P, (DR / 8) * 2, PB, 8, TILE, NS, BF);
  }
  if (!ok) return cudaErrorInvalidValue;
  TcArgs args;
  args.q_cat = static_cast<const uint16_t*>(q_cat);
  args.plan = plan;
  args.pages = pg;
  args.page_table = page_table;
  args.part_o = part_o;
  args.seg_cap = seg_cap;
  args.part_lse = part_lse;
  args.err = err;
  args.B = Bv;
  args.max_pages = max_pages;
  args.num_pages = num_pages;
  args.scale_log2 = scale * 1.4426950408889634f;
  args.qs = qs;
  args.q_rows = q_rows;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = launch_config(workers, s, attr);
  auto go = [&](auto kernel, size_t smem) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cfg.dynamicSmemBytes = smem;
    return cudaLaunchKernelEx(&cfg, kernel, m[0], m[1], m[2], m[3], m[4], tq_pe, args);
  };
  if (fmt == MLA_FMT_BF16) return go(attend_tc_kernel<MLA_FMT_BF16>, smem_bytes<MLA_FMT_BF16>());
  if (fmt == MLA_FMT_INT8) return go(attend_tc_kernel<MLA_FMT_INT8>, smem_bytes<MLA_FMT_INT8>());
  return go(attend_tc_kernel<MLA_FMT_INT4>, smem_bytes<MLA_FMT_INT4>());
}

}  // namespace mla
