/*
 * tahq.h -- C ABI of the GB300 (sm_103a) TAH-Quant activation codec.
 *
 * The codec compresses the [tokens x channels] activation tensor that one pipeline
 * stage sends to the next and restores it on the receiving stage, as described in
 * "TAH-Quant: Effective Activation Quantization in Pipeline Parallelism over Slow
 * Network" (arXiv 2506.01352v2), §3.1-§3.5 and Algorithm 1 (stage a sends
 * Q(a(xi)), stage b de-quantises it).
 *
 * Conventions shared by every entry point
 *   - The caller owns all memory.  Tensor, output and workspace pointers are DEVICE
 *     pointers on the current CUDA device; the library allocates nothing.
 *   - Calls are asynchronous and ordered on `stream` (a cudaStream_t passed as void*,
 *     NULL = the legacy default stream).  The return code covers host-side argument
 *     checks and kernel-launch errors only.
 *   - Errors found on the device (non-finite input, a bounded wait that gave up, an
 *     inconsistent select, a bit width outside 1..8, a stream shorter than its slots)
 *     set bits of a 32-bit status word at the head of the workspace.  The word is
 *     cleared at the start of every call and read by tahq_get_device_status().  No
 *     kernel traps or waits without a bound.
 *   - Layout: x and out are row-major [tokens, channels].  Tile t covers channels
 *     [w*tile, (w+1)*tile) of token t / (channels/tile), w = t % (channels/tile).
 *   - Alignment: x, out and codes 16 B; workspace 256 B; scales, zeros 4 B.
 *   - Limits: tile a power of two in 8..128 dividing channels (so pivots fit a byte and
 *     every slot is whole bytes); hblock a power of two in 2..tile; 1 <= bits_lo <
 *     bits_hi <= 8; bits_lo <= budget <= bits_hi; tokens_per_group divides tokens
 *     (0 = one group of all tokens) and a group holds fewer than 2^31 tiles;
 *     tokens * channels < 2^40.
 */
#ifndef TAHQ_H
#define TAHQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    TAHQ_OK = 0,
    TAHQ_ERR_ARG = 1,          /* an argument is outside the limits above             */
    TAHQ_ERR_UNSUPPORTED = 2,  /* valid for the method, not built here (e.g. tile 96) */
    TAHQ_ERR_WORKSPACE = 3,    /* workspace missing, misaligned or too small          */
    TAHQ_ERR_CUDA = 4,         /* a CUDA runtime call or kernel launch failed         */
    TAHQ_ERR_DEVICE_STATUS = 5 /* the device status word is non-zero                  */
} tahq_status;

typedef enum { TAHQ_F32 = 0, TAHQ_BF16 = 1 } tahq_dtype;

/* Bits of the device status word. */
#define TAHQ_DEV_NONFINITE 0x1u          /* an input tile sum or key was not finite     */
#define TAHQ_DEV_WAIT_TIMEOUT 0x2u       /* a cross-block wait gave up after its bound  */
#define TAHQ_DEV_SELECT_MISMATCH 0x4u    /* candidate count disagreed with histogram    */
#define TAHQ_DEV_BAD_BITS 0x8u           /* decode: a bit width outside 1..8 or pivot   */
#define TAHQ_DEV_STREAM_OVERRUN 0x10u    /* decode: slots run past codes_bytes          */
#define TAHQ_DEV_BAD_WIRE 0x20u          /* decode_wire: header differs from the args   */

/*
 * Exact size in bytes of the packed code stream for these parameters.  §3.4: the
 * mixed-precision payload is a contiguous uint8 stream of a fixed shape.  Each group of
 * tokens_per_group tokens has n_g = tokens_per_group * channels / tile tiles, of which
 * K = floor((budget - bits_lo) * n_g / (bits_hi - bits_lo)) carry bits_hi and the rest
 * bits_lo, so every group occupies n_g*tile*bits_lo/8 + K*tile*(bits_hi-bits_lo)/8 bytes.
 * Returns 0 for invalid arguments (and for tokens == 0).
 */
size_t tahq_payload_size(int64_t tokens, int64_t channels, int tile, int bits_lo, int bits_hi,
                         float budget, int64_t tokens_per_group);

/* Number K of tiles per group that receive bits_hi (formula above); -1 if invalid. */
int64_t tahq_hi_count(int64_t tokens, int64_t channels, int tile, int bits_lo, int bits_hi,
                      float budget, int64_t tokens_per_group);

/*
 * Bytes of device workspace tahq_encode needs for these parameters (status word,
 * per-group entropy histograms, select candidates, per-tile keys, scan words).
 * Returns 0 for invalid arguments.  The workspace may be reused by later calls on the
 * same stream; calls that overlap on the device must not share a workspace.
 */
size_t tahq_workspace_size(int64_t tokens, int64_t channels, int tile, int hblock, int bits_lo,
                           int bits_hi, float budget, int64_t tokens_per_group);

/*
 * Encode x (dtype f32 or bf16, [tokens, channels]) -- §3.1-§3.4:
 *   per tile: entropy key (§3.2 eq. (1)-(2), Shannon sign), outlier ratio r (§3.3
 *   eq. (3), tau = 2.0) and pivot d = first arg-max |x|;
 *   per group: the K tiles of highest (key, then lowest tile index) get bits_hi (§3.2
 *   "Top-p% tile selection"), the others bits_lo;
 *   per tile: if r > tau, swap positions 0 and d and apply the Sylvester Hadamard
 *   transform to every hblock-wide block, scaled by 1/sqrt(hblock) (§3.3 eq. (4));
 *   then min/max asymmetric quantisation to b bits (round to nearest even) and
 *   LSB-first packing into the tile's slot; slots follow each other in tile order.
 * Outputs (device, caller-allocated):
 *   codes  [tahq_payload_size(...)] bytes
 *   scales [n_tiles] fp32  step (max-min)/(2^b-1), 0 for a constant tile
 *   zeros  [n_tiles] fp32  tile minimum (the de-quantisation offset)
 *   bits   [n_tiles] u8    bits_lo or bits_hi
 *   pivots [n_tiles] u8    d for transformed tiles, 0xFF otherwise
 * n_tiles = tokens * channels / tile.  Returns TAHQ_ERR_ARG / _UNSUPPORTED /
 * _WORKSPACE before launching anything, TAHQ_ERR_CUDA on a launch failure.
 */
tahq_status tahq_encode(const void *x, tahq_dtype dtype, int64_t tokens, int64_t channels, int tile,
                        int hblock, int bits_lo, int bits_hi, float budget,
                        int64_t tokens_per_group, uint8_t *codes, float *scales, float *zeros,
                        uint8_t *bits, uint8_t *pivots, void *workspace, size_t workspace_bytes,
                        void *stream);

/*
 * tahq_encode with two of the method's parameters as arguments.
 *   tau: the outlier threshold ("TAH-Quant" §3.3 eq. (3); its Appendix F compares
 *     tau = 0, 2, 4 and infinity).  A tile is transformed when
 *     r = |a(1)| / (|a(2)| + 1e-12) > tau (fp32 IEEE division, strict): tau = 0
 *     transforms every tile whose r is above zero, tau = INFINITY none.  The entropy keys,
 *     and so the widths, do not depend on tau.  Negative or NaN: TAHQ_ERR_ARG.
 *   alloc_tile: the allocation tile A of §3.2 "Tile decomposition" (0 = tile, the pages'
 *     default; A = channels is the token-level allocation).  One entropy key per A
 *     consecutive channels of a token (the key over its A values, same canonical order),
 *     ranked per group; K = floor((budget - bits_lo) * n_A / (bits_hi - bits_lo)) of the
 *     group's n_A = tokens_per_group * channels / A allocation tiles get bits_hi, and every
 *     tile takes its allocation tile's width; the outlier test, transform and quantiser
 *     stay per tile.  A must be a power-of-two multiple of tile dividing channels
 *     (else TAHQ_ERR_ARG) and A * sizeof(element) <= 32768 (else TAHQ_ERR_UNSUPPORTED).
 *     The payload is then tahq_payload_size_ex's; tahq_workspace_size is enough for any A.
 * tau = 2.0f, alloc_tile = 0 is tahq_encode.  Same arguments, layouts, ownership and
 * errors as tahq_encode otherwise.
 */
tahq_status tahq_encode_ex(const void *x, tahq_dtype dtype, int64_t tokens, int64_t channels,
                           int tile, int hblock, int bits_lo, int bits_hi, float budget,
                           int64_t tokens_per_group, float tau, int alloc_tile, uint8_t *codes,
                           float *scales, float *zeros, uint8_t *bits, uint8_t *pivots,
                           void *workspace, size_t workspace_bytes, void *stream);

/* Payload bytes with allocation tiles of alloc_tile channels (0 = tile); 0 if invalid. */
size_t tahq_payload_size_ex(int64_t tokens, int64_t channels, int tile, int alloc_tile,
                            int bits_lo, int bits_hi, float budget, int64_t tokens_per_group);

/* Bytes of device workspace tahq_decode needs; 0 for invalid arguments. */
size_t tahq_decode_workspace_size(int64_t tokens, int64_t channels, int tile);

/*
 * Decode -- the inverse path of §3.3 ("apply H_G^T to the de-quantised values") and
 * Algorithm 1 step 5: unpack each tile's codes from its slot (slot offsets are the
 * running sum of tile*bits[t]/8 in tile order, so no group structure is needed),
 * v = fma(q, scale, zero); if pivots[t] != 0xFF: Hadamard per hblock block, scale
 * 1/sqrt(hblock), swap positions 0 and pivots[t].  out is fp32 [tokens, channels].
 * codes_bytes bounds every read of codes: a stream shorter than its slots sets
 * TAHQ_DEV_STREAM_OVERRUN (the affected tiles decode to 0) instead of reading past it.
 */
tahq_status tahq_decode(const uint8_t *codes, size_t codes_bytes, const float *scales,
                        const float *zeros, const uint8_t *bits, const uint8_t *pivots,
                        int64_t tokens, int64_t channels, int tile, int hblock, float *out,
                        void *workspace, size_t workspace_bytes, void *stream);

/*
 * Size of the fixed device scratch array behind tahq_decode_noalloc: 256 KiB, held in
 * the memory of every GPU that loads the library until the process exits.  It bounds
 * the shapes that entry point accepts: tahq_decode_workspace_size(tokens, channels,
 * tile) must not exceed it, i.e. at most 52288 decode chunks (4 bytes each, plus 8 bytes
 * per 8 chunks) -- about 6.7 M tiles of width 128, 13.4 M of width 64, 26.8 M of width 32,
 * 53.5 M of width 16, 107 M of width 8.
 */
#define TAHQ_NOALLOC_SCRATCH_BYTES (256u * 1024u)

/*
 * tahq_decode for callers that cannot allocate device memory at all -- for example a
 * receiving stage whose runtime plans every device buffer in advance and gives the codec
 * only its inputs and outputs, or a C caller with no device allocator, for which a
 * cudaMalloc inside the receive loop would also stall the whole device.  (The paper has
 * no counterpart to this entry point: it is a packaging choice of this library.)
 * Same arguments and results as tahq_decode, minus the workspace: the scratch comes from
 * a fixed array inside the library (TAHQ_NOALLOC_SCRATCH_BYTES).  Nothing is allocated:
 * no cudaMalloc, no cudaFree, no allocating library call.
 *   - The first call on each device looks up the array's device address (with that
 *     device current) and caches it; make that first call before any stream capture.
 *   - Shapes that need more scratch than the array holds are rejected with
 *     TAHQ_ERR_WORKSPACE before anything is launched.
 *   - Every call on a device shares the one array.  Each call clears the part it uses
 *     first, but calls whose work overlaps on the GPU (other streams, other host threads)
 *     race on it: order them on one stream or use tahq_decode with separate workspaces.
 *   - device_status (device pointer, may be NULL) receives a copy of the call's device
 *     status word (TAHQ_DEV_* bits) when the decode kernel has finished, ordered on
 *     `stream`.
 */
tahq_status tahq_decode_noalloc(const uint8_t *codes, size_t codes_bytes, const float *scales,
                                const float *zeros, const uint8_t *bits, const uint8_t *pivots,
                                int64_t tokens, int64_t channels, int tile, int hblock,
                                float *out, uint32_t *device_status, void *stream);

/*
 * WIRE FORMAT ("TAH-Quant" §3.2: the 1-bit per-tile width map travels with the payload
 * as metadata; §3.4: heterogeneous precisions and metadata in one contiguous uint8 byte
 * stream of fixed size per shape; the pages count about 0.61 metadata bits per element at
 * a tile of 64, i.e. 39 bits a tile).  One buffer, sections at 16-byte boundaries:
 *   [0, 128)      header, little-endian: u32 magic "TAHQ", u16 version 1, u16 128,
 *                 i64 tokens, i64 channels, i64 tokens per group, u16 tile, u16 hblock,
 *                 u8 bits_lo, u8 bits_hi, u8 pivot bits pb = log2(tile), u8 0, f32 budget,
 *                 f32 tau, u64 tiles, u64 offsets of the four sections below, u64 payload
 *                 bytes, u64 total bytes, zeros;
 *   width map     bit t (LSB first) = tile t has bits_hi;
 *   metadata      per tile a u32: fp16 scale in bits 0-14 with the transform flag in bit
 *                 15 (a scale is never negative), fp16 zero in bits 16-31;
 *   pivots        pb bits per tile (LSB first), the pivot of a transformed tile, else 0;
 *   payload       the packed slots of tahq_encode (same layout, same size);
 * padding bytes are zero.  Widths and transform decisions are those of tahq_encode_ex;
 * the quantiser rounds to the wire's fp16 metadata: zero = the largest fp16 value <= the
 * tile minimum, scale = the smallest fp16 value s >= 0 with zero + (2^b - 1) s >= the tile
 * maximum (exact arithmetic), codes RNE((v - zero) * RN(1 / s)) (0 when s = 0), decode
 * fmaf(q, s, zero).  Inputs beyond the fp16 range (|v| > 65504) give undefined codes.
 */

/* Bytes of the wire buffer for these parameters (fixed by the shape); 0 if invalid. */
size_t tahq_wire_size(int64_t tokens, int64_t channels, int tile, int bits_lo, int bits_hi,
                      float budget, int64_t tokens_per_group);

/* Device workspace of tahq_encode_wire (the encoder's plus four per-tile arrays). */
size_t tahq_wire_workspace_size(int64_t tokens, int64_t channels, int tile, int hblock,
                                int bits_lo, int bits_hi, float budget, int64_t tokens_per_group);

/* Device workspace of tahq_decode_wire (the decoder's plus four per-tile arrays). */
size_t tahq_wire_decode_workspace_size(int64_t tokens, int64_t channels, int tile);

/*
 * Encode x (as tahq_encode_ex, same arguments and threshold tau) into the wire buffer
 * `wire` (device, 16-byte aligned, at least tahq_wire_size bytes; the caller owns it).
 * Returns the errors of tahq_encode_ex, TAHQ_ERR_ARG for a missing, misaligned or short
 * buffer, TAHQ_ERR_WORKSPACE for a workspace below tahq_wire_workspace_size.
 */
tahq_status tahq_encode_wire(const void *x, tahq_dtype dtype, int64_t tokens, int64_t channels,
                             int tile, int hblock, int bits_lo, int bits_hi, float budget,
                             int64_t tokens_per_group, float tau, uint8_t *wire,
                             size_t wire_bytes, void *workspace, size_t workspace_bytes,
                             void *stream);

/*
 * Decode a wire buffer into out [tokens * channels] fp32 (device, 16-byte aligned).  The
 * arguments are those the buffer was encoded with (they fix its layout); a header that
 * differs from them (tau aside) sets TAHQ_DEV_BAD_WIRE in the workspace's status word,
 * and invalid fields set the bits tahq_decode sets.  Host-side errors as tahq_decode.
 */
tahq_status tahq_decode_wire(const uint8_t *wire, size_t wire_bytes, int64_t tokens,
                             int64_t channels, int tile, int hblock, int bits_lo, int bits_hi,
                             float budget, int64_t tokens_per_group, float *out, void *workspace,
                             size_t workspace_bytes, void *stream);

/* ---- the backward pass's gradient codec ----------------------------------------------
 * "TAH-Quant" §3.5 and Algorithm 1 (the second stage sends a fixed-point quantisation of
 * the gradient with respect to the activations back to the first; 6-8 bits, 10 after the
 * NaN event of Appendix H) and Appendix H eq. (24) (g_hat = Q(c g) / c).  The §3.3
 * asymmetric quantizer at one width `bits` (1..16) on tiles of `tile` consecutive channels
 * of a token, no bit allocation, no outlier transform: per tile zero = min, scale =
 * RN((max - min) / Q), codes RNE((v - min) * RN(Q / (max - min))), Q = 2^bits - 1 (scale 0
 * and codes 0 when max - min < 2^-120), v = RN(scale_c * g); decode
 * RN(fma(q, scale, zero) / scale_c).  scale_c must be a positive power of two (exact
 * scaling).  Codes are packed least significant bit first at `bits` bits, tile after tile
 * (tile * bits / 8 bytes each); scales and zeros hold one fp32 value per tile.
 */

/* Bytes of the packed codes; 0 for invalid arguments or a tile other than 32, 64, 128. */
size_t tahq_naive_codes_bytes(int64_t tokens, int64_t channels, int tile, int bits);

/*
 * Encode grad [tokens * channels] fp32 (device, 16-byte aligned) into codes (device,
 * 16-byte aligned, tahq_naive_codes_bytes), scales and zeros (device, tokens * channels /
 * tile floats each).  All memory is the caller's; stream-ordered, no synchronisation.
 * TAHQ_ERR_ARG: bits outside 1..16, channels not a multiple of tile, scale_c not a
 * positive power of two, a NULL or misaligned pointer; TAHQ_ERR_UNSUPPORTED: tile other
 * than 32, 64 or 128; TAHQ_ERR_CUDA: a launch failed.
 */
tahq_status tahq_naive_encode(const float *grad, int64_t tokens, int64_t channels, int tile,
                              int bits, float scale_c, uint8_t *codes, float *scales,
                              float *zeros, void *stream);

/* Decode into out [tokens * channels] fp32 (device, 16-byte aligned); errors as encode. */
tahq_status tahq_naive_decode(const uint8_t *codes, const float *scales, const float *zeros,
                              int64_t tokens, int64_t channels, int tile, int bits,
                              float scale_c, float *out, void *stream);

/*
 * Copy the device status word of the last call that used `workspace` into *status_out
 * (may be NULL) after synchronising `stream` (only that stream).  Returns TAHQ_OK if
 * the word is zero, TAHQ_ERR_DEVICE_STATUS if not, TAHQ_ERR_CUDA if the copy failed.
 */
tahq_status tahq_get_device_status(const void *workspace, uint32_t *status_out, void *stream);

/*
 * TAH-Quant on a gradient with the scaling of eq. (24) (TAH-Quant Appendix H, Table 10:
 * the activation codec applied to backward gradients; eq. (24): g_hat = Q(c g) / c).
 *
 * tahq_encode_scaled: the codec of tahq_encode_ex (tau as there, allocation tile = tile)
 * applied to RN(scale_c * x), with scale_c a positive finite power of two (so the scaling
 * is exact unless scale_c * x leaves the normal float range; bf16 inputs stay bf16).  The
 * outputs describe scale_c * x: scales and zeros are those of the scaled values.  On the
 * streaming encoder's shapes (tau = 2, tiles of 32..128 values, groups of whole 32 KB
 * input chunks) the kernels read the scaled values directly; otherwise a scaled copy of x
 * is written into the workspace after the codec's own part.  Either way the workspace
 * must hold tahq_scaled_workspace_size() bytes (0 on invalid arguments).
 * tahq_decode_scaled: tahq_decode with every output value RN(value / scale_c) (the
 * decoder multiplies by 1 / scale_c as it stores; the same workspace as tahq_decode).  Errors as for tahq_encode / tahq_decode; a scale_c that is not a
 * positive finite power of two gives TAHQ_ERR_ARG.
 */
size_t tahq_scaled_workspace_size(int64_t tokens, int64_t channels, int tile, int hblock,
                                  int bits_lo, int bits_hi, float budget,
                                  int64_t tokens_per_group, tahq_dtype dtype);
tahq_status tahq_encode_scaled(const void *x, tahq_dtype dtype, int64_t tokens, int64_t channels,
                               int tile, int hblock, int bits_lo, int bits_hi, float budget,
                               int64_t tokens_per_group, float tau, float scale_c,
                               uint8_t *codes, float *scales, float *zeros, uint8_t *bits,
                               uint8_t *pivots, void *workspace, size_t workspace_bytes,
                               void *stream);
tahq_status tahq_decode_scaled(const uint8_t *codes, size_t codes_bytes, const float *scales,
                               const float *zeros, const uint8_t *bits, const uint8_t *pivots,
                               int64_t tokens, int64_t channels, int tile, int hblock,
                               float scale_c, float *out, void *workspace,
                               size_t workspace_bytes, void *stream);

/*
 * Exercises the bounded wait that every cross-block wait of the kernels uses (the pages
 * have no counterpart: this is the codec's own failure detection).  One thread waits in
 * turn on eight counters in `workspace` that nothing advances, each wait limited to
 * limit_ns nanoseconds of the device's global timer; the first gives up after the limit
 * and sets TAHQ_DEV_WAIT_TIMEOUT in the status word, and the others return at once on
 * seeing it.  workspace: device memory of at least 1024 bytes, 256-byte aligned (an
 * encode workspace serves; its first 1024 bytes are cleared first); elapsed_ns: device
 * pointer to two uint64 (may be NULL) that receive the time spent in the waits and the
 * number of waits that gave up.  Stream-ordered; read the result with
 * tahq_get_device_status(workspace, ...).  limit_ns must be in 1 .. 10^10.
 */
tahq_status tahq_test_wait_timeout(void *workspace, size_t workspace_bytes, uint64_t limit_ns,
                                   uint64_t *elapsed_ns, void *stream);

/* Human-readable name of a tahq_status value (static string, never NULL). */
const char *tahq_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int tahq_version(void);

/*
 * The host-side tables the kernels use for the canonical base-2 logarithm
 * (lg x = e + fmaf(P(r), r, T[i]), r = fmaf(m, R[i], -1) for x = 2^e m, i = the top 7
 * fraction bits of m, P(r) = fmaf(fmaf(k[2], r, k[1]), r, k[0])):
 * R[i] = nearest float to 1/(1 + i/128), T[i] = nearest float to -log2(R[i]),
 * k[j] = nearest float to (-1)^j / ((j+1) ln 2), j = 0..2.  Exposed so that a CPU test
 * can check them without a GPU.  T and R hold 128 floats, k 3.
 */
void tahq_log2_tables(float *T, float *R, float *k);

#ifdef __cplusplus
}
#endif

#endif /* TAHQ_H */
