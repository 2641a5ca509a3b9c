/*
 * mmq.h -- C ABI of the GB300 (sm_103a) prefill quantized matrix multiply (MMQ):
 * k-quant weight super-blocks (q6_K 210 B, q4_K 144 B, 256 values each) times
 * per-32 q8 activations,
 *
 *     q6_K: Y[t,j] = sum_c sum_h d_a[t,c] * (d*sc[2(c%8)+h]) * I[t,j,c,h]
 *     q4_K: Y[t,j] = sum_c d_a[t,c] * ((d*sc_c) * I[t,j,c] - (dmin*m_c) * ssum[t,c])
 *
 * (d, sc, dmin, m from the weight super-block; d_a, ssum the activation chunk's
 * scale and code sum)
 *
 * with I the integer dot of a 16-value (q6_K) or 32-value (q4_K) sub-block.
 *
 * Sources (page title, section):
 *   [r45] "r45 - cp.async for the q6_K A-side staging: mechanism confirmed,
 *          wall-neutral (REVERTED)"
 *   [r56] "r56 - q6_K A-side bundle: A cp.async + W_dsc f32 plane (LANDED)"
 *   [r58] "r58 - q4_K BT spec + cp.async-db2 transplant (REVERTED)"
 * The pages show the registration step, the activation prepass and the GEMM
 * launch ([r56] §3.1: registration gates and planes; [r45] §1.1: the
 * quantize-transpose prepass; [r58] §2.2: the GEMM's staging); this ABI exposes
 * those three steps as calls.
 *
 * Conventions (all calls):
 *  - Every buffer pointer is a DEVICE pointer owned by the caller.  The library
 *    never allocates or frees device memory; sizes come from the *_bytes queries.
 *  - Calls are asynchronous on stream `s` (NULL = legacy default stream).
 *    Argument, shape and alignment errors are returned synchronously, before
 *    anything is launched; a failed launch returns MMQ_ERR_CUDA.
 *  - K = id must be a multiple of 256 (one super-block); od >= 1 may be odd; M >= 1.
 *  - Buffers read by bulk copies (qa, scales, packed) must be 16-byte aligned,
 *    else MMQ_ERR_ALIGN.  x and Y need 4-byte alignment.
 *  - Every bounded wait inside a kernel gives up after about two seconds, sets the
 *    library's one sticky device error word (one per device) and lets the kernel
 *    exit; mmq_get_device_error() reports and clears it, whichever kernel set it.
 *    Results of a launch that timed out are undefined, and so are those of launches
 *    queued after it until the word is cleared (their waits give up early once they
 *    see it set).
 *  - Calls may come from several host threads; the one piece of shared host
 *    state is the label mmq_last_path() returns (the most recent GEMM launch
 *    of the process).
 */
#ifndef MMQ_GB300_H
#define MMQ_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (the runtime's stream handle). */
typedef struct CUstream_st* mmq_stream_t;

typedef enum {
    MMQ_OK = 0,
    MMQ_ERR_ARG = 1,         /* null pointer, bad type id, ldx < K, ldy < od */
    MMQ_ERR_SHAPE = 2,       /* K/id not a multiple of 256, M/od < 1, sizes over the limits */
    MMQ_ERR_ALIGN = 3,       /* a pointer is not aligned as stated above */
    MMQ_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
    MMQ_ERR_TIMEOUT = 5,     /* a bounded in-kernel wait expired (see mmq_get_device_error) */
    MMQ_ERR_UNSUPPORTED = 6  /* no sm_103 device is current */
} mmq_status;

typedef enum { MMQ_Q4_K = 12, MMQ_Q6_K = 14 } mmq_type;

/* Size limits (checked; MMQ_ERR_SHAPE beyond them). */
#define MMQ_MAX_M (1 << 22)
#define MMQ_MAX_OD (1 << 22)
#define MMQ_MAX_ID (1 << 20)

/* --------------------------------------------------------------------------
 * Activation planes ([r45] §2.3 and [r56] §1: the prepass writes a
 * pre-transposed q8 code plane and a d/ssum scale pair per (chunk, token),
 * padded token rows zero-filled).
 *
 * Layout (fixed, documented so a caller can read it back):
 *   Mp = 128 * ceil(M/128) padded tokens; nkb = K/64; nchunk = K/32; nsb = K/256.
 *   qa:     Mp*K f16 values, the q8 codes held as exact binary16 integers
 *           (zero as +0).
 *           Tile (mt, kb) = tokens 128*mt.. and values 64*kb.. is a 16384-byte
 *           block at byte (mt*nkb + kb)*16384.  Inside it token r (0..127) and
 *           value k (0..63) sit at byte r*128 + (((k/8) ^ (r%8))*16) + (k%8)*2
 *           (the 128-byte swizzle of the tensor-core operand tile).
 *   scales: two planes (offsets from mmq_act_scale_layout):
 *     pairs  Mp*nchunk entries of 8 bytes {float d, int32 ssum}; entry (t, c) at
 *            index ((t/128)*nchunk + c)*128 + t%128.
 *     am     the q4_K min-term operand ma = d*ssum (one f32 multiply) split into
 *            tf32 hi = round-to-nearest(ma) and lo = round-to-nearest(ma - hi):
 *            per (token tile mt, super-block sb) an 8192-byte block at
 *            (mt*nsb + sb)*8192 holding the hi tile then the lo tile, each
 *            128 rows x 8 chunks of 4-byte values, row r / chunk k at byte
 *            (r/8)*256 + (k/4)*128 + (r%8)*16 + (k%4)*4.
 *   Rows t >= M hold code 0, d 0, ssum 0, ma 0.
 *   qa, M <= MMQ_SMALL_M only: after the Mp*K*2 bytes of tiles, the same codes
 *     as int8, M rows of K bytes, each group of 8 values stored in the order
 *     (0,2,4,6,1,3,5,7): value k of token t at byte t*K + (k & ~7) +
 *     ((k & 7) >> 1) + 4*(k & 1).  The weight-streaming GEMM reads this plane.
 *     mmq_act_plane_bytes includes it in qa_bytes.
 *   M <= MMQ_FT_MAX_M only (offsets from mmq_act_ft_layout), the few-token GEMM's
 *     activation operand, with N = 16*ceil(M/16):
 *     tq (in qa, after the int8 plane if any) per k-block kb a 2*N*128-byte block
 *        at kb*2*N*128: N rows of hi then N rows of lo, row t / value k at byte
 *        t*128 + (((k/8) ^ (t%8))*16) + (k%8)*2 (f16), where for the token's
 *        super-block p = 2^(P-127), P = min(260 - E, 253) and E the f32 exponent
 *        field of the largest of its 8 chunk scales d, s = p*d (exact),
 *        s_hi = rn_f16(s), s_lo = rn_f16(s - s_hi), and for each code q:
 *        hi = rn_f16(s_hi*q), lo = rn_f16(fma(s_hi, q, -hi) + s_lo*q) (f16 fma);
 *     ip (in scales, after am) f32 1/p at index sb*MMQ_FT_MAX_M + t (t < N);
 *     fm (in scales, after ip) f32 ma = d*ssum (one f32 multiply) of chunk c of
 *        super-block sb at index (sb*8 + c % 8)*MMQ_FT_MAX_M + t (t < N).
 * -------------------------------------------------------------------------- */
#define MMQ_SMALL_M 8
#define MMQ_FT_MAX_M 64
mmq_status mmq_act_plane_bytes(int M, int K, size_t* qa_bytes, size_t* scale_bytes);
mmq_status mmq_act_scale_layout(int M, int K, size_t* pair_offset, size_t* pair_bytes,
                                size_t* am_offset, size_t* am_bytes);
/* Offsets and sizes of the few-token planes (all six 0 when M > MMQ_FT_MAX_M). */
mmq_status mmq_act_ft_layout(int M, int K, size_t* tq_offset, size_t* tq_bytes,
                             size_t* ip_offset, size_t* ip_bytes, size_t* fm_offset, size_t* fm_bytes);

/* Quantize x [M][ldx] f32 (row-major, first K values of each row used) per
 * 32-value chunk: d = amax/127 (IEEE f32 division), q = round(x/d) (IEEE f32
 * division, ties away from zero, clamped to [-127,127]; d == 0 gives q = 0),
 * ssum = sum q.  Writes qa and scales in the layout above.  x must be finite. */
mmq_status mmq_quantize_act(const float* x, int M, int K, int ldx,
                            void* qa, void* scales, mmq_stream_t s);

/* --------------------------------------------------------------------------
 * Registration-time weight repack ([r56] §2.2-§2.3 W_dsc plane: exact f16->f32
 * and int->f32 conversions, one f32 multiply, no FMA contraction; chunk-major
 * so one tile's window is contiguous; [r58] §5 names the same plane for q4_K;
 * [r56] §1 and [r58] §3.2: codes unpacked once at registration).
 *
 * For q6_K the pack calls then read FLAG word 0 back to the host and return only
 * when the stream has finished the pack (not while the stream is being captured
 * into a graph); the GEMM calls on that buffer use it to choose their kernel.  The
 * choice affects the speed only: every kernel reads FLAG itself.
 *
 * raw_blocks: od rows x id/256 super-blocks, row-major, 210 B (q6_K: ql[128]@0,
 *   qh[64]@128, int8 scales[16]@192, f16 d@208) or 144 B (q4_K: f16 d@0,
 *   f16 dmin@2, scales[12]@4 = 16 six-bit fields little-endian, fields 0..7 the
 *   scales sc_c and 8..15 the mins m_c, qs[128]@16).  Code of value e:
 *   q6_K ((ql[e/2] >> 4*(e%2)) & 15 | ((qh[e/4] >> 2*(e%4)) & 3) << 4) - 32,
 *   q4_K (qs[e/2] >> 4*(e%2)) & 15.  Value e of a q6_K block uses scales[e/16].
 *
 * packed (caller-owned, mmq_packed_weight_bytes() bytes) holds ten planes at
 * the offsets mmq_packed_weight_layout() returns; Np = 128*ceil(od/128),
 * nkb = id/64, nchunk = id/32, nsb = id/256; rows j >= od are zero:
 *   CODES  Np*id f16 integers in 16384-byte tiles (nt, kb) at (nt*nkb + kb)*16384,
 *          row r / value k at byte r*128 + (((k/8) ^ (r%8))*16) + (k%8)*2.
 *          The integer sub-block scale is folded into the code, exactly: q4_K
 *          sc_c*q (|.| <= 945); q6_K sc*q when every |scales[i]| of the tensor is
 *          <= 64 (|.| <= 2048), else sc*l with l = (q + 32) & 15 (|.| <= 1920) and
 *          the second tile in CODES2.
 *   PAIRS  Np*nchunk entries of two floats, entry (j, c) at index
 *          ((j/128)*nchunk + c)*128 + j%128:
 *            q6_K {d*scales[2*(c%8)], d*scales[2*(c%8)+1]}
 *            q4_K {d*sc_(c%8), dmin*m_(c%8)}
 *   SBD    f32 d per (row, super-block) at index ((j/128)*nsb + sb)*128 + j%128.
 *   AUX    per (row tile nt, super-block sb) an 8192-byte block at (nt*nsb + sb)*8192:
 *            q4_K: dmn = dmin*m_c split exactly into tf32 hi + lo; the hi tile then
 *                  the lo tile, row r / chunk k at (r/8)*256 + (k/4)*128 + (r%8)*16 + (k%4)*4;
 *            q6_K: the 16 scales as f32, scale s of row r at byte (s*128 + r)*4
 *                  (kept for read-back; no kernel reads it).
 *   FLAG   q6_K: uint32 word 0 = 1 if CODES are folded, word 1 = max |scales[i]|.
 *   RAW    the raw blocks re-laid for the weight-streaming GEMM, od rows x nsb
 *          blocks, row-major: q4_K 144 B [qs[128] | d | dmin | scales[12]],
 *          q6_K 224 B [ql[128] | qh[64] | scales[16] | d | 14 zero bytes].
 *   CW     compact codes for the few-token GEMM, which widens them to f16 in
 *          tensor memory: per (nt, kb) W = 2 (q4_K) or 4 (q6_K) words of 16 bytes
 *          per row, word-major: word w of row r at ((nt*nkb + kb)*W + w)*2048 + r*16.
 *          q4_K: word w holds chunk 2*kb + w, the 4-bit code of value 8u + 2p + h
 *          of the chunk (u, p = 0..3, h = 0,1) at bit 4p + 16h of its 32-bit word u.
 *          q6_K: word w holds the 16 values of sub-block w of the k-block, one byte
 *          4*(q + 32) each, value 4u + o (u, o = 0..3) at byte 2*(o & 1) + (o >> 1)
 *          of its 32-bit word u.
 *   SC     sub-block scales per (nt, sb): 16 bytes per row at ((nt*nsb + sb)*128 + r)*16:
 *          q4_K the six-bit sc_0..sc_7 then m_0..m_7, one per byte; q6_K scales[16].
 *   DM     q4_K: f32 dmin per (row, super-block) at index ((j/128)*nsb + sb)*128 + j%128
 *          (the few-token GEMM's min-term factor); q6_K: empty.
 *   CODES2 q6_K: Np*id f16 values in the CODES tile layout, 16*sc*(h - 2) with
 *          h = (q + 32) >> 4 (a multiple of 16 of magnitude <= 4096, exact) when
 *          CODES holds sc*l, so that CODES + CODES2 = sc*q; zero when CODES is
 *          folded; q4_K: empty.
 * -------------------------------------------------------------------------- */
typedef enum {
    MMQ_PLANE_CODES = 0,
    MMQ_PLANE_PAIRS = 1,
    MMQ_PLANE_SBD = 2,
    MMQ_PLANE_AUX = 3,
    MMQ_PLANE_FLAG = 4,
    MMQ_PLANE_RAW = 5,
    MMQ_PLANE_CW = 6,
    MMQ_PLANE_SC = 7,
    MMQ_PLANE_DM = 8,
    MMQ_PLANE_CODES2 = 9,
    MMQ_NUM_WEIGHT_PLANES = 10
} mmq_weight_plane;

mmq_status mmq_packed_weight_bytes(mmq_type t, int od, int id, size_t* bytes);
mmq_status mmq_packed_weight_layout(mmq_type t, int od, int id, size_t offsets[MMQ_NUM_WEIGHT_PLANES],
                                    size_t sizes[MMQ_NUM_WEIGHT_PLANES]);
mmq_status mmq_pack_weights(mmq_type t, const void* raw_blocks, int od, int id,
                            void* packed, mmq_stream_t s);

/* Fused registration of two weights that read the same input ([r58] §5, the fused
 * FFN gate/up GEMM): packs raw_a (od_a rows) and raw_b (od_b rows), both of type t
 * and width id, as ONE weight of od = od_a + od_b rows in the layout above, rows
 * [0, od_a) from raw_a and [od_a, od) from raw_b; the planes equal those of
 * mmq_pack_weights on the two raw buffers concatenated row-wise, without that copy.
 * One GEMM on it (mmq_gemm_* with od = od_a + od_b) over one set of activation
 * planes writes both outputs side by side: Y[t][j] for j < od_a is row j of a,
 * Y[t][od_a + j] row j of b.  packed must hold mmq_packed_weight_bytes(t, od, id).
 * MMQ_ERR_SHAPE for od_a or od_b < 1 or a sum over MMQ_MAX_OD; otherwise as
 * mmq_pack_weights. */
mmq_status mmq_pack_weights_fused(mmq_type t, const void* raw_a, int od_a, const void* raw_b, int od_b, int id,
                                  void* packed, mmq_stream_t s);

/* GGUF interop (registration time): nblocks q4_K (144 B) or q6_K (210 B) blocks in
 * the public ggml (llama.cpp) block layout, rewritten into the layout documented
 * above for raw_blocks, so that mmq_pack_weights can take weights read from a GGUF
 * file.  The byte offsets of d, dmin, scales and the code arrays are the same in
 * both; what moves is the position of each code and the q4_K scale packing:
 *   ggml q4_K: value 64j+l (l < 32) = low nibble of qs[32j+l], value 64j+32+l = its
 *     high nibble; sub-block s < 4: sc = S[s] & 63, m = S[s+4] & 63; s >= 4:
 *     sc = (S[s+4] & 15) | (S[s-4] >> 6) << 4, m = (S[s+4] >> 4) | (S[s] >> 6) << 4
 *     (S = scales[12]);
 *   ggml q6_K: value 128n+32p+l: low 4 bits = nibble p/2 of ql[64n+32(p%2)+l],
 *     high 2 bits = bits 2p..2p+1 of qh[32n+l]; scales[16] and d unchanged.
 * src and dst are device pointers (any alignment); dst == src converts in place;
 * other overlaps are undefined.  nblocks = 0 is a no-op.  MMQ_ERR_ARG for a bad
 * type or a null pointer. */
mmq_status mmq_convert_ggml_blocks(mmq_type t, const void* src, size_t nblocks, void* dst, mmq_stream_t s);

/* --------------------------------------------------------------------------
 * The GEMM: Y[t][j] (t < M, j < od, row stride ldy floats) is overwritten with
 * the formula at the top of this file.  packed comes from mmq_pack_weights of
 * the same (type, od, id); qa/scales from mmq_quantize_act with K = id and the
 * same M.  Four kernels compute it (mmq_last_path names the one launched;
 * mmq_debug_select_large_m_kernel can force a choice):
 *  - M <= MMQ_SMALL_M (decode and tail shapes), the weight-streaming kernel,
 *    except where the few-token kernel below is faster (measured crossovers,
 *    w = od*id: q4_K with w >= 2^24 and M >= 7, or w >= 2^25 and M >= 5; q6_K
 *    with w >= 2^25 and M >= 4): the
 *    RAW plane and the int8 activation plane, exact integer dots on the CUDA
 *    cores (dp4a), and the scales applied per chunk in the formula's own order
 *    (q4_K: Y += d_a*(d*sc_c*I) - (d_a*ssum)*(dmin*m_c); q6_K: Y +=
 *    d_a*(d*sc0*I_0 + d*sc1*I_1)), with a fixed reduction order;
 *  - otherwise for M <= MMQ_FT_MAX_M, the few-token kernel: the CW codes are
 *    widened to exact f16 integers (q4_K sc*q; q6_K sc*q when FLAG says every
 *    |scales[i]| <= 64, else the two exact tiles sc*l/4 and 4*sc*(h-2), l and h
 *    the low 4 and high 2 bits of q + 32) in tensor memory and contracted on
 *    tcgen05 against the tq operand (f16 hi and lo of p*d_a*q_a as one 2N-row
 *    operand), one f32 accumulator per stage, then d and 1/p applied per
 *    super-block; the q4_K min term sum_c (dmin*m_c)*(d_a*ssum) from DM, SC and
 *    fm in f32 FMAs (each token's sum over c = 0..7 in order); when the weight
 *    tiles are few, each is split along K over a
 *    cluster of up to 8 CTAs whose partial sums are added in rank order
 *    (deterministic);
 *  - larger M, the super-block kernel or the chunk kernel below, whichever a
 *    round-count cost model of both, fitted to GB300 timings, expects to finish
 *    first (mmq_debug_route gives the choice; q6_K whose registration found the
 *    codes in two tiles always takes the chunk kernel).  The super-block kernel:
 *    the activation operand p*d_a*q_a as an f16 hi + lo pair
 *    (about 2^-21 relative per value) times the exact f16 CODES (and CODES2 for
 *    two-tile q6_K, a second pair of MMAs into the same accumulator), summed over
 *    a whole super-block in f32, then d and 1/p per super-block.  In both tile
 *    kernels, when the last round of tiles fills at most half the SMs (or all
 *    tiles do), those tiles run as two K-halves added into Y after a zeroing
 *    kernel, 0 + a + b, the same in either order;
 *  - the chunk kernel: the integer dots sum_chunk (sc*q)*q_a run
 *    exactly (codes held as f16 integers, two-tile q6_K as two MMAs per 16
 *    values, every partial sum an integer below 2^24 in the f32 accumulator)
 *    and the f32 scales are applied per chunk (d_a) and per super-block (d).
 * The super-block and chunk kernels compute the q4_K min term sum_c
 * (d_a*ssum)*(dmin*m_c) as a tf32 hi/lo tensor-core contraction (relative error
 * about 2^-21 per product), each TMEM accumulator covering at most 64
 * super-blocks before it is added into Y's f32 sums.
 * Y is deterministic for given inputs and kernel.  Rows t >= M and columns
 * j >= od are never written.  ldy >= od.
 * -------------------------------------------------------------------------- */
mmq_status mmq_gemm_q6k(const void* packed, int od, int id, const void* qa, const void* scales,
                        int M, float* Y, int ldy, mmq_stream_t s);
mmq_status mmq_gemm_q4k(const void* packed, int od, int id, const void* qa, const void* scales,
                        int M, float* Y, int ldy, mmq_stream_t s);

/* Debug/verification: the same GEMM kernel (same staging, same tensor-core
 * contraction) writes the raw integer dots it accumulates instead of Y, as f32
 * values holding the exact integers, at dots[(t*od + j)*nsub + s]:
 *   q4_K: nsub = id/32, s = chunk c: sc_c * sum(q * q_a)
 *   q6_K: nsub = id/32, s = chunk c: sc0*I_0 + sc1*I_1
 * (I_h = sum(q * q_a) over the chunk's 16-value half h; |value| < 2^24). */
mmq_status mmq_debug_gemm_dots(mmq_type t, const void* packed, int od, int id, const void* qa,
                               const void* scales, int M, float* dots, mmq_stream_t s);

/* Debug/verification, host logic only (no CUDA call): the kernel the default
 * selection of mmq_gemm_* gives for (t, od, id, M) on a device with nsm SMs, for
 * q6_K codes folded (fold = 1), in two tiles (0) or of unknown state (-1, taken as
 * folded; q4_K ignores fold): *kernel = 0 weight-streaming, 1 chunk, 2 super-block,
 * 3 few-token.  MMQ_ERR_ARG for a null kernel, nsm < 1 or fold outside -1..1;
 * otherwise the shape errors of the GEMM calls. */
mmq_status mmq_debug_route(mmq_type t, int od, int id, int M, int fold, int nsm, int* kernel);

/* Debug/verification: which kernel computes Y (process-wide).
 *   0 (default): as described above the GEMM calls;
 *   1: the chunk kernel for every M > MMQ_SMALL_M (128-token tiles);
 *   2: the super-block kernel for every M > MMQ_SMALL_M;
 *   3: as 0, but the few-token kernel never splits a tile over a CTA cluster;
 *   4: as 0, but the few-token kernel also for M <= MMQ_SMALL_M.
 * Returns MMQ_ERR_ARG for any other value.  Not thread-safe against GEMM calls
 * in flight on other host threads. */
mmq_status mmq_debug_select_large_m_kernel(int which);

/* Debug/verification of the timeout path (a loud error, never a silent wrong
 * result: [r56] §3.1).  Arms a one-shot injection for the next GEMM launch that
 * runs a tile kernel (M > MMQ_SMALL_M): its waits give up after limit_ns
 * (1 us .. 2 s) instead of about two seconds, and the producer of its first CTA
 * leaves operand fill number `fill` (0-based, counted over that CTA's k-blocks)
 * out, so the wait for it runs out, the launch exits early and
 * mmq_get_device_error() then returns MMQ_ERR_TIMEOUT (and clears the word).
 * That launch takes no CTA-cluster split.  Its Y is undefined.  fill < 0
 * disarms a pending injection.  MMQ_ERR_ARG for a limit outside the range.
 * Process-wide host state; no CUDA call. */
mmq_status mmq_debug_inject_wait_timeout(int fill, unsigned long long limit_ns);

/* Synchronizes `s`, then reports and clears the sticky device error word:
 * MMQ_ERR_TIMEOUT if a bounded wait expired since the last call, MMQ_ERR_CUDA
 * if the synchronization failed, else MMQ_OK. */
mmq_status mmq_get_device_error(mmq_stream_t s);

const char* mmq_status_string(mmq_status st);

/* Label of the path the most recent GEMM launch took (liveness check,
 * [r56] §3.2 and §4: a fast path needs a visible label because parity alone
 * cannot show it ran). */
const char* mmq_last_path(void);

/* Number of kernel launches the library has made in this process (every entry
 * point that launches adds the kernels it launched: prepass 1, repack 4 or 5,
 * GEMM 1, or 2 when K-half tiles are first zeroed). */
unsigned long long mmq_launch_count(void);

/* Library version string. */
const char* mmq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MMQ_GB300_H */
