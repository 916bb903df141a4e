/*
 * qmoe.h -- C ABI of the GB300 (sm_103a) fused decode-and-multiply library for
 * sub-2-bit compressed mixture-of-experts expert weights.
 *
 * Two stored formats are supported:
 *
 *  1. Dictionary-coded ternary weights (QMoE).  Every weight of a row is one of
 *     {0, -s, +s} with one fp16 scale s per row.  Rows are cut into blocks of
 *     `block` weights; each block is a sequence of 16-bit codewords, each of
 *     which indexes a shared 2^16-entry dictionary whose entry expands to 2..28
 *     ternary values (whole pairs).  Source: the QMoE paper-summary page,
 *     sections "The Fixed-to-Variable Dictionary Code" (Algorithm 1 and
 *     Figure 4) and "The GPU Decoding Kernel" (Listing 1 and "Encoding").
 *
 *  2. Residual vector quantisation after a two-sided randomized Hadamard
 *     transform.  Source: "Quantization as Cache Amplification", section
 *     "Codec" (incoherence processing and residual vector quantization), with
 *     the runtime sign order of "M8.5 - Extreme Weight Compression and
 *     Representations", section 0x06H.
 *
 * Conventions for every entry point:
 *  - Return value: QMOE_OK (0) or a negative qmoe_status.  Arguments are
 *    validated on the host before anything is launched; a failed call
 *    launches nothing.  qmoe_last_error() gives a message for the calling
 *    thread's last failure.
 *  - "device" pointers are CUDA device (or managed) memory; "host" pointers
 *    are ordinary process memory.  The caller owns every buffer; no entry
 *    point allocates or frees device memory, and scratch space comes from a
 *    caller-provided workspace whose size the matching *_ws_size call returns.
 *  - Device work is enqueued on `stream` (a cudaStream_t, NULL = the legacy
 *    default stream) and is asynchronous: outputs are valid once the stream
 *    has reached the call.  Kernels that detect a corrupt stream (a codeword
 *    expanding past its block, a block that does not expand to its length)
 *    record QMOE_EFORMAT in a device error word and keep going with clamped
 *    indices; qmoe_check_status() reads and clears that word.  Nothing traps.
 *  - bf16 / fp16 values are passed as their 16-bit patterns.
 *  - Matrices are row-major with rows = output features: y = W x.
 */
#ifndef QMOE_H
#define QMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QMOE_OK = 0,
    QMOE_EINVAL = -1,        /* bad argument: null pointer, size, shape, range */
    QMOE_ECAPACITY = -2,     /* output or workspace buffer too small */
    QMOE_ECUDA = -3,         /* a CUDA runtime call failed */
    QMOE_EFORMAT = -4,       /* corrupt codeword stream or dictionary */
    QMOE_ETIMEOUT = -5,      /* a bounded device wait gave up */
    QMOE_EUNSUPPORTED = -6   /* valid request this build does not implement */
} qmoe_status;

#define QMOE_DICT_ENTRIES 65536
#define QMOE_DICT_WORDS (2 * QMOE_DICT_ENTRIES)
#define QMOE_MAX_RUN 28
/* bytes of the kernel-private compact dictionary made by qmoe_dict_compact */
#define QMOE_COMPACT_BYTES (7 * QMOE_DICT_ENTRIES)
#define QMOE_RVQ_DIM 8
#define QMOE_RVQ_CODES 256
/* most residual stages an RVQ code may have */
#define QMOE_RVQ_MAX_STAGES 3
/* code formats of an rvq_matrix_set */
#define QMOE_VQ_RVQ 0 /* residual k-means codebooks: one 8-bit index per stage */
#define QMOE_VQ_E8P 1 /* E8P lattice code: one 16-bit word per 8-vector */
/* entries of the E8P base table (absolute patterns) */
#define QMOE_E8P_PATTERNS 256

/* ======================================================================
 * Host-side codec (dictionary format)
 * ====================================================================== */

/*
 * Algorithm 1 (QMoE page, "Dictionary generation"): the 2^16 most probable
 * sequences of 1..14 ternary pairs under the independence model
 * P(0) = p0, P(w_min) = P(w_max) = (1 - p0)/2, most probable first.  The
 * priority of a sequence is n0*ln(p0) + nz*ln((1-p0)/2) from its counts;
 * equal priorities are ordered by the symbol tuple, lexicographically,
 * shorter prefix first.
 *
 *  symbols   host int8 {-1,0,+1}, n values, or NULL.  When given, p0 is
 *            measured as the zero fraction of these weights; when NULL the
 *            argument p0 is used.
 *  p0        zero probability in (0, 1) (ignored when symbols != NULL).
 *  dict_words host out, QMOE_DICT_WORDS uint32: entry e is the pair
 *            (dict_words[2e], dict_words[2e+1]) in the Figure 4 layout:
 *            bits [3:0] of both words = pair count; word h holds symbol
 *            14h+i at bits [5+2i:4+2i]; symbol 0 = zero, 1 = w_min (-s),
 *            2 = w_max (+s); unused fields are 0.
 *  p0_used   host out (may be NULL): the p0 the dictionary was built for.
 * Errors: EINVAL (null output, p0 outside (0,1), n == 0 with symbols given,
 * a measured p0 of 0 or 1).
 */
int qmoe_encode_dictionary(const int8_t* symbols, size_t n, double p0,
                           uint32_t* dict_words, double* p0_used);

/*
 * Greedy longest-match encoder (QMoE page, "Encoding (compression time)"):
 * each row of a rows x cols ternary matrix is cut into blocks of `block`
 * weights (the last block of a row may be shorter); inside a block the
 * encoder repeatedly emits the codeword of the longest dictionary entry that
 * is a prefix of the remaining weights.  Codewords never cross a block.
 *
 *  tern      host int8 [rows][cols] in {-1,0,+1}.
 *  cols, block  even, > 0.
 *  dict_words host, QMOE_DICT_WORDS uint32 (qmoe_encode_dictionary layout).
 *  codes     host out uint16 [codes_cap], or NULL to only count.
 *  n_codes   host out: number of codewords of the whole matrix.
 *  blk_off   host out uint32 [rows * ceil(cols/block) + 1] (may be NULL when
 *            codes is NULL): index of the first codeword of block b of row r
 *            at [r*nb + b]; the last element is the total.
 * Errors: EINVAL (shape, null, value outside {-1,0,1}), ECAPACITY (codes_cap
 * smaller than the count; *n_codes still holds the count), EFORMAT (the
 * dictionary cannot express some block: it lacks a ternary pair).
 * Thread-safe: several threads may pack different matrices at once.
 */
int qmoe_pack(const int8_t* tern, int rows, int cols, int block,
              const uint32_t* dict_words, uint16_t* codes, size_t codes_cap,
              size_t* n_codes, uint32_t* blk_off);

/*
 * Derive the kernel-private compact dictionary from the canonical entries.
 * The compact table holds, per entry, the pair count and the positions and
 * signs of its nonzero weights in 24 bits (a uint16 plane followed by a
 * uint8 plane): three 6-bit slots for entries with up to three nonzeros,
 * four 4-bit slots (and a flag) for entries with four nonzeros all in their
 * first eight positions (the four-nonzero entries of dictionaries for
 * p0 >= 0.8); any other entry carries a flag that sends the kernels to its
 * canonical words.  A third plane repeats each entry as one uint32 (the
 * uint16 entry in bits 0-15, the uint8 entry in bits 16-23) for kernels that
 * read the table from global memory: one gather per codeword instead of two.
 * Upload the result
 * next to the canonical words and point qmoe_dict.compact at it.
 *  dict_words host in, QMOE_DICT_WORDS uint32.
 *  compact   host out, QMOE_COMPACT_BYTES bytes.
 * Errors: EINVAL (null), EFORMAT (pair counts of the two halves disagree, a
 * pair count outside 1..14, symbol value 3, or a nonzero in an unused field).
 */
int qmoe_dict_compact(const uint32_t* dict_words, void* compact);

/* ======================================================================
 * Device descriptors
 * ====================================================================== */

typedef struct {
    const uint32_t* words;   /* device, QMOE_DICT_WORDS canonical uint32 */
    const void* compact;     /* device, QMOE_COMPACT_BYTES from qmoe_dict_compact */
} qmoe_dict;

/*
 * Device encoder: the greedy longest-match encoding of qmoe_pack on the GPU,
 * with the same codewords and block offsets bit for bit (QMoE page,
 * "Encoding (compression time)"; the page encodes on the host, one thread per
 * row).  One GPU thread encodes one (row, block) against a hash table of the
 * dictionary that the call builds in the workspace; a scan of the per-block
 * counts gives the offsets.  Asynchronous on `stream`.
 *
 *  dict      device descriptor; only dict->words is read.
 *  tern      device int8 [rows][cols] in {-1,0,+1}.
 *  rows >= 0; cols, block even, > 0.
 *  codes     device out uint16 [codes_cap].  rows*cols/2 codewords always
 *            suffice; the exact count is blk_off[rows*nb] once the stream has
 *            reached the end of the call.
 *  blk_off   device out uint32 [rows*nb + 1], nb = ceil(cols/block): the
 *            qmoe_pack layout.
 *  workspace device scratch of qmoe_pack_device_ws_size() bytes (a 3 MB
 *            dictionary table plus rows*nb*block bytes); caller-owned, not
 *            shared by concurrent calls.
 * Errors on the host: EINVAL (shape, NULL), ECAPACITY (workspace too small),
 * ECUDA.  Errors found on the device go to the error word that
 * qmoe_check_status() returns: EINVAL (a weight outside {-1,0,1}, more than
 * 2^32 codewords), EFORMAT (bad dictionary entry, or a block the dictionary
 * cannot express), ECAPACITY (more codewords than codes_cap: the excess is
 * dropped).
 */
int qmoe_pack_device_ws_size(int rows, int cols, int block, size_t* bytes);
int qmoe_pack_device(const qmoe_dict* dict, const int8_t* tern, int rows, int cols, int block,
                     uint16_t* codes, size_t codes_cap, uint32_t* blk_off, void* workspace,
                     size_t ws_bytes, void* stream);

/*
 * `count` dictionary-coded matrices of the same shape (e.g. the wi matrices
 * of all experts of a layer), with their block offsets stored compactly (a
 * re-encoding of qmoe_pack's uint32 offsets that qmoe_offsets_compact
 * makes; the rate ledger counts these stored widths):
 *  - row_off[e*(rows+1) + r]: index of the first codeword of row r of matrix
 *    e, relative to code_base[e]; row_off[e*(rows+1) + rows] = its codeword
 *    count.  uint32.
 *  - blk_len[(e*rows + r)*(nb-1) + b], b < nb-1: the number of codewords of
 *    block b of row r (the last block's count is what the row leaves),
 *    nb = ceil(cols/block).  uint8: a block holds at most block/2 <= 255
 *    codewords, so block <= 510.
 * Matrix e's codewords start at codes[code_base[e]]; its scales are
 * scale_f16[e*rows + r].  code_base may be NULL when count == 1 (base 0).
 * The kernels read codewords in aligned 16-byte chunks: `codes` must be
 * 16-byte aligned and its allocation must extend (zero-padded) to the next
 * multiple of 8 codewords after the last codeword of the set.  Offsets must
 * lie inside the codes allocation; the kernels check that each row and each
 * block expands to exactly its length (QMOE_EFORMAT otherwise) but cannot
 * check offsets against the allocation size.
 */
typedef struct {
    const uint16_t* codes;      /* device */
    const uint64_t* code_base;  /* device [count], or NULL when count == 1 */
    const uint32_t* row_off;    /* device [count][rows + 1] */
    const uint8_t* blk_len;     /* device [count][rows][nb - 1] (NULL when nb == 1) */
    const uint16_t* scale_f16;  /* device [count][rows] fp16 bits */
    int count, rows, cols, block;
} qmoe_matrix_set;

/*
 * The compact offsets of qmoe_matrix_set from qmoe_pack's (or the device
 * encoder's) block offsets of one matrix: row_off[r] = blk_off[r*nb],
 * row_off[rows] = blk_off[rows*nb]; blk_len[r*(nb-1) + b] =
 * blk_off[r*nb + b + 1] - blk_off[r*nb + b] for b < nb-1.
 *  blk_off  host in uint32 [rows*nb + 1], non-decreasing from 0.
 *  row_off  host out uint32 [rows + 1];  blk_len host out uint8
 *           [rows*(nb-1)] (may be NULL when nb == 1).
 * Errors: EINVAL (null pointer, rows < 1, nb < 1), EFORMAT (offsets that
 * decrease, do not start at 0, or a block of more than 255 codewords).
 */
int qmoe_offsets_compact(const uint32_t* blk_off, int rows, int nb,
                         uint32_t* row_off, uint8_t* blk_len);

/* ======================================================================
 * Dictionary path: fused decode-and-multiply
 * ====================================================================== */

/*
 * y[t][r] = s_r * sum_c w_rc x[t][c] for t < T: the expert matrix-vector
 * product (T = 1) and its skinny-GEMM generalisation with an inner loop over
 * tokens (QMoE page, "The GPU Decoding Kernel" and the proposed fix for
 * batched experts in the limitations section).  Weights are decoded in
 * registers; dense weights are never written to memory.
 *  mat       host pointer to a descriptor with count == 1.
 *  x_bf16    device bf16 [T][cols].
 *  y         device [T][rows], fp32 when y_is_f32 else bf16 (nearest even).
 * Accumulation is fp32; the row scale multiplies the accumulated sum once.
 * Errors: EINVAL (shape, null, count != 1, odd cols/block), ECUDA.
 */
int qmoe_expert_matvec(const qmoe_dict* dict, const qmoe_matrix_set* mat,
                       const void* x_bf16, int T, void* y, int y_is_f32,
                       void* stream);

/*
 * Router (step a1): top-k of router logits and softmax gates.
 *  logits  device fp32 [T][E];  ids out device int32 [T][k] (descending
 *  logit, equal logits to the lower id);  gates out device fp32 [T][k] =
 *  softmax over all E logits read at the chosen experts (not renormalised).
 * Errors: EINVAL (k < 1, k > E, k > 32, E > 8192), ECUDA.
 */
int qmoe_route(const float* logits, int T, int E, int k, int32_t* ids,
               float* gates, void* stream);

/*
 * Bucketiser (step a2): stable counting sort of the flat slots t*k + j by
 * expert ids[t][j].  counts[E], offsets[E+1] (exclusive prefix sum) and
 * perm[T*k] (slots of expert e, increasing, at perm[offsets[e]..]) are
 * device int32 outputs.  Ids outside [0, E) make the call record
 * QMOE_EINVAL in the device error word and drop those slots.
 */
int qmoe_bucketise(const int32_t* ids, int T, int k, int E, int32_t* counts,
                   int32_t* offsets, int32_t* perm, void* stream);

/* Workspace bytes for qmoe_moe_layer with these shapes. */
int qmoe_moe_layer_ws_size(int E, int d_model, int d_ff, int T, int k,
                           size_t* bytes);

/*
 * Which dictionary kernel a qmoe_moe_layer call with these shapes launches for
 * each of its two matrices (host only, no device work): QMOE_KERNEL_FLAT, the
 * flat-stream CUDA-core kernel (a warp decodes a run of rows as one codeword
 * stream; compact table in shared memory); QMOE_KERNEL_ROWS, the
 * row-per-lane CUDA-core kernel (a lane walks one row; compact table in
 * shared memory), taken when a job's rows fill the block's warps in nearly
 * whole rounds; QMOE_KERNEL_FLAT_L2, the flat-stream kernel reading the
 * compact table through L1/L2 (calls with fewer than 16 token slots).  *tc is
 * 1 when the call also launches the tensor-core kernel for experts with at
 * least 32 tokens (calls with at least 256 token slots).  Both CUDA-core
 * kernels compute the same sums (QMoE page, "The GPU Decoding Kernel"); they
 * differ in how work is spread.
 * Errors: EINVAL (bad sizes or NULL outputs), EUNSUPPORTED (d_model or d_ff
 * too large for the staged activations).
 */
#define QMOE_KERNEL_FLAT 0
#define QMOE_KERNEL_ROWS 1
#define QMOE_KERNEL_FLAT_L2 2
int qmoe_moe_layer_kernels(int E, int d_model, int d_ff, int T, int k,
                           int* wi_kernel, int* wo_kernel, int* tc);

/*
 * Switch-Transformer-shaped MoE feed-forward layer on dictionary-coded
 * experts: for every token t and slot j with expert e = ids[t][j],
 *   h = bf16(relu(Wi_e x_t)),  o = Wo_e h,  y_t = sum_j gates[t][j] * o
 * (slots summed in order).  Experts that receive no token are skipped.
 *  wi        count = E, rows = d_ff, cols = d_model.
 *  wo        count = E, rows = d_model, cols = d_ff.
 *  x_bf16    device bf16 [T][d_model];  ids device int32 [T][k];
 *  gates     device fp32 [T][k];  y device [T][d_model] fp32 or bf16.
 *  workspace device, ws_bytes >= qmoe_moe_layer_ws_size(...).
 * Errors: EINVAL, ECAPACITY (workspace), ECUDA.
 */
int qmoe_moe_layer(const qmoe_dict* dict, const qmoe_matrix_set* wi,
                   const qmoe_matrix_set* wo, const void* x_bf16, int T, int k,
                   const int32_t* ids, const float* gates, void* y,
                   int y_is_f32, void* workspace, size_t ws_bytes,
                   void* stream);

/*
 * qmoe_moe_layer without a workspace argument.  The paper has no counterpart:
 * this entry point exists for callers that cannot allocate device memory,
 * such as code hosted inside a framework that owns all device memory through
 * its own pool, or serving loops that forbid cudaMalloc/cudaFree after
 * start-up because those calls can synchronise the device.  It computes
 * exactly what qmoe_moe_layer computes, with the same arguments minus the
 * workspace, and allocates nothing: its scratch is a file-scope device array
 * of 16 MiB (16 << 20 bytes) that every GPU loading the library holds until
 * the process exits.
 *  - The first call on a device looks up the array's address on that device
 *    (with that device current), and looks it up again in another context
 *    or after a device reset; make that first call before any stream
 *    capture.
 *  - Calls whose needs (qmoe_moe_layer_ws_size) exceed 16 MiB are rejected
 *    with QMOE_ECAPACITY and launch nothing.
 *  - All calls share the array, which keeps the last call's contents; no
 *    scratch byte needs to start at zero.  Calls that overlap on the GPU
 *    (other streams, other host threads) race on the array: serialise them.
 * Errors: as qmoe_moe_layer, plus ECAPACITY for an oversize call.
 */
int qmoe_moe_layer_noalloc(const qmoe_dict* dict, const qmoe_matrix_set* wi,
                           const qmoe_matrix_set* wo, const void* x_bf16,
                           int T, int k, const int32_t* ids,
                           const float* gates, void* y, int y_is_f32,
                           void* stream);

/* ======================================================================
 * Residual-VQ path
 * ====================================================================== */

/*
 * `count` RVQ-coded matrices of the same shape.  Matrix e has S_e residual
 * stages (2 for every matrix unless `stages` is given):
 *  idx       device uint8: matrix e's codes start at idx + idx_base[e]
 *            (idx_base NULL: at e*rows*(cols/8)*2) and are [rows][cols/8][S_e]
 *            codebook indices of each 8-weight vector of the rotated weight,
 *            stage 1 first;
 *  codebooks device fp16 bits [n_stages][256][8] shared by the whole set;
 *  scale_f16 device [count][rows] fp16 per-row scales;
 *  sign_out  device int8 [count][rows] (+1/-1), sign_in [count][cols];
 *  stages    device uint8 [count], each in 1 .. n_stages, or NULL (all 2);
 *  idx_base  device uint64 [count] byte offsets, or NULL;
 *  n_stages  codebooks in the set (0 means 2), at most QMOE_RVQ_MAX_STAGES.
 * Frequency-conditioned allocation ("Quantization as Cache Amplification",
 * Frequency-Conditioned Bit Allocation) gives popular experts more stages;
 * see rvq_stage_allocation.  rows and cols are powers of two (2 .. 8192),
 * cols a multiple of 8.  Decoded rotated weight: W'[r][8v+j] =
 * fp32(s_r) * (((fp32(C1[i1][j]) + fp32(C2[i2][j])) + fp32(C3[i3][j])) ...),
 * the adds left to right over the matrix's stages; layer output
 * y = D_out H_rows (W' (H_cols D_in x)) with H the normalised Walsh-Hadamard
 * matrix.  Zero-initialising the last four fields gives the two-stage set.
 *
 * format QMOE_VQ_E8P ("M8.5 - Extreme Weight Compression and
 * Representations", 0x06E): the same transforms and per-row scales, and
 *  idx       device uint16 code words, little-endian, [rows][cols/8] per
 *            matrix (2 bytes per vector: the offsets above with S_e = 2);
 *  codebooks device uint32 [256]: the base table of e8p_base_table;
 *  stages    NULL and n_stages 0.
 * Code word c decodes to the 8-vector v: pattern p = c & 255, nibble j of
 * table[p] is 2|a_j| (1, 3 or 5); coordinate j < 7 is negative when bit 8+j
 * is set, coordinate 7 when that makes sum_j s_j |a_j| odd otherwise (so the
 * sum is even: a point of D8 + 1/2); v_j = s_j |a_j| + (bit 15 ? 1/4 : -1/4).
 * Decoded rotated weight: W'[r][8v+j] = fp32(s_r) * v_j (exact in fp32).
 */
typedef struct {
    const uint8_t* idx;
    const uint16_t* codebooks;
    const uint16_t* scale_f16;
    const int8_t* sign_out;
    const int8_t* sign_in;
    int count, rows, cols;
    const uint8_t* stages;
    const uint64_t* idx_base;
    int n_stages;
    int format; /* QMOE_VQ_RVQ (0) or QMOE_VQ_E8P */
} rvq_matrix_set;

/* Workspace bytes for rvq_expert_matmul. */
int rvq_expert_matmul_ws_size(int rows, int cols, int T, size_t* bytes);

/*
 * y[t] = D_out H (W' (H D_in x_t)) for one RVQ-coded matrix (count == 1):
 * input transform, fused codebook decode + multiply (CUDA cores for T < 16,
 * tcgen05 tensor cores with fp16 operands and fp32 accumulation for
 * T >= 16), output transform.  On the tensor-core path each rotated
 * activation row is first multiplied by a power of two that brings its
 * largest magnitude into [2^14, 2^15) (undone exactly in the epilogue), then
 * split into an fp16 high part and the fp16 of the remainder; any finite bf16
 * input stays inside fp16's range, and values below 2^-25 of their row's
 * largest one are the only ones that lose low bits.
 *  x_bf16 device bf16 [T][cols];  y device [T][rows] fp32 or bf16.
 * Errors: EINVAL, ECAPACITY, ECUDA.
 */
int rvq_expert_matmul(const rvq_matrix_set* mat, const void* x_bf16, int T,
                      void* y, int y_is_f32, void* workspace, size_t ws_bytes,
                      void* stream);

/* Workspace bytes for rvq_moe_layer. */
int rvq_moe_layer_ws_size(int E, int d_model, int d_ff, int T, int k,
                          size_t* bytes);

/*
 * OLMoE-shaped SwiGLU MoE layer on RVQ-coded experts: for every token t and
 * slot j with expert e = ids[t][j],
 *   h = bf16(silu(gate_e x_t) * up_e x_t),  o = down_e h,
 *   y_t = sum_j gates[t][j] * o  (slots in order),
 * each of gate/up/down applied through its own transforms as in
 * rvq_expert_matmul.  gate and up: rows = d_ff, cols = d_model; down:
 * rows = d_model, cols = d_ff; all with count = E.
 * Errors: EINVAL, ECAPACITY, ECUDA.
 */
int rvq_moe_layer(const rvq_matrix_set* gate, const rvq_matrix_set* up,
                  const rvq_matrix_set* down, const void* x_bf16, int T, int k,
                  const int32_t* ids, const float* gates, void* y,
                  int y_is_f32, void* workspace, size_t ws_bytes,
                  void* stream);

/*
 * Host-side RVQ encoder for one matrix: rotated weight W' = H_rows D_out W
 * D_in H_cols (float64 butterflies, each transform divided by sqrt(n) at the
 * end), per-row scale fp16(sqrt(sum_c W'^2 / cols)) with the sum taken left
 * to right, u = W'/s cut into 8-vectors, i1 = nearest stage-1 codeword,
 * i2 = nearest stage-2 codeword to u - C1[i1] (squared distance summed over
 * j = 0..7 in order, ties to the lower index).
 *  w        host float64 [rows][cols];  sign_out/sign_in host int8 +-1;
 *  codebooks host fp16 bits [2][256][8];  idx host out uint8
 *  [rows][cols/8][2];  scale_f16 host out [rows].
 * Errors: EINVAL (shape: powers of two, cols % 8; null; a zero row).
 */
int rvq_pack(const double* w, int rows, int cols, const int8_t* sign_out,
             const int8_t* sign_in, const uint16_t* codebooks, uint8_t* idx,
             uint16_t* scale_f16);

/*
 * rvq_pack with n_stages residual stages (1 .. QMOE_RVQ_MAX_STAGES): stage s
 * takes the codeword of codebooks[s] nearest to what stages 1 .. s-1 leave
 * of u (float64 residuals).  codebooks host fp16 bits [n_stages][256][8];
 * idx host out uint8 [rows][cols/8][n_stages].  rvq_pack is n_stages = 2.
 */
int rvq_pack_stages(const double* w, int rows, int cols, const int8_t* sign_out,
                    const int8_t* sign_in, const uint16_t* codebooks, int n_stages,
                    uint8_t* idx, uint16_t* scale_f16);

/*
 * Stages per expert for an average of s_bar ("Quantization as Cache
 * Amplification", Frequency-Conditioned Bit Allocation, rank-based form):
 * the floor(E/3) most popular experts get s_bar + 1 stages, the floor(E/3)
 * least popular s_bar - 1, the others s_bar, so the mean rate is s_bar.
 * Equal popularity ranks the lower expert id as more popular.
 *  popularity host float64 [E] (any positive weights, e.g. activation
 *             frequencies);  stages host out uint8 [E].
 * Errors: EINVAL (NULL, E < 1, s_bar - 1 or s_bar + 1 outside
 * 1 .. QMOE_RVQ_MAX_STAGES when E >= 3).
 */
int rvq_stage_allocation(const double* popularity, int E, int s_bar, uint8_t* stages);

/*
 * The E8P base table ("M8.5 - Extreme Weight Compression and
 * Representations", 0x06E: 8 bits select one of 256 stored absolute
 * patterns, 1 KiB): the 256 patterns a in {1/2, 3/2, 5/2, ...}^8 of smallest
 * squared norm, equal norms in lexicographic order of (2a_0, .., 2a_7);
 * entry p holds 2a_j in bits 4j .. 4j+3.
 *  table host out uint32 [256].  Errors: EINVAL (NULL).
 */
int e8p_base_table(uint32_t* table);

/*
 * Host-side E8P encoder for one matrix: the rotated weight W' as in rvq_pack,
 * per-row scale s_r = fp16(sqrt(sum_c W'^2 / cols) / kappa) (sum left to
 * right; kappa^2 = 2450/2048, the mean power per coordinate of the 65 536
 * codewords), u = W'/s_r cut into 8-vectors, and for each the code word of
 * the nearest codeword (squared distance summed over j = 0..7 in float64;
 * ties to the smaller code word).
 *  w host float64 [rows][cols];  sign_out/sign_in host int8 +-1;
 *  codes host out uint16 [rows][cols/8];  scale_f16 host out [rows].
 * Errors: EINVAL (shape: powers of two, cols % 8; null; a zero row).
 */
int e8p_pack(const double* w, int rows, int cols, const int8_t* sign_out,
             const int8_t* sign_in, uint16_t* codes, uint16_t* scale_f16);

/*
 * The encoder's search alone: for each of n 8-vectors u (host float64
 * [n][8]) the code word of the nearest E8P codeword, as in e8p_pack.
 *  codes host out uint16 [n].  Errors: EINVAL (NULL with n > 0, non-finite u).
 */
int e8p_nearest(const double* u, size_t n, uint16_t* codes);

/* ======================================================================
 * Status and test exports
 * ====================================================================== */

/*
 * Measurement hook (the pages have no counterpart: it exists for timing).
 * When `events` is non-NULL, later qmoe_moe_layer and rvq_moe_layer calls in
 * this process record events[i] (cudaEvent_t handles owned by the caller) on
 * their stream at phase boundaries:
 *   qmoe_moe_layer: [0] start, [1] after planning, [2] after the wi
 *                   CUDA-core kernel, [3] after the wi tensor-core kernel,
 *                   [4] after the wo CUDA-core kernel, [5] after the wo
 *                   tensor-core kernel (and the combine when k > 1) = end.
 *   rvq_moe_layer:  [0] start, [1] after planning and the input transform,
 *                   [2] after the gate and up kernels, [3] after SwiGLU and the
 *                   down input transform, [4] after the down kernel, [5] end.
 * n must be at least 6 (NULL/0 turns the hook off).  Process-wide and not
 * thread-safe.  Errors: EINVAL.
 */
int qmoe_set_phase_events(void* const* events, int n);

/* Synchronises `stream`, returns and clears the device error words
 * (QMOE_OK, QMOE_EFORMAT, QMOE_EINVAL, QMOE_ECAPACITY or QMOE_ETIMEOUT), or
 * QMOE_ECUDA. */
int qmoe_check_status(void* stream);

/* Message describing the calling thread's last failed call ("" if none). */
const char* qmoe_last_error(void);

/* Test export: decoded dictionary-coded weights, device fp32 [rows][cols]
 * (count == 1).  Every block is checked to expand to exactly its length. */
int qmoe_decode_dense(const qmoe_dict* dict, const qmoe_matrix_set* mat,
                      float* w_out, void* stream);

/* Test export: decoded rotated RVQ or E8P weight W', device fp32
 * [rows][cols] (count == 1). */
int rvq_decode_dense(const rvq_matrix_set* mat, float* w_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* QMOE_H */
