// Host-side launchers of the library's kernels.  Each returns a cudaError_t
// value as int (0 = queued fine).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dflash {

// ---- init-time quantisers / packers (k_quant.cu)
int q4_quantize_pack(const float* w_dev, int N, int K, uint8_t* packed, int tile0, int ksteps, __half* scale_scratch,
                     cudaStream_t st);
int q4_unpack(const uint8_t* packed, int tile0, int N, int K, int ksteps, int8_t* codes, uint16_t* scales,
              cudaStream_t st);
int i8_rows_quantize_pack(const float* w_dev, int N, int K, int Npad, int ksteps, int8_t* packed, float* row_scale,
                          cudaStream_t st);
int i8_unpack(const int8_t* packed, int N, int K, int ksteps, int8_t* codes, cudaStream_t st);

// ---- matmuls (k_gemm.cu)
// Activation operand of the quantised matmuls: int8 codes held as exact f16
// integers, [rows][ld] with ld >= K (K a multiple of 64), one f32 scale a row.
struct QAct {
    const __half* codes;
    const float* scale;
    int ld;
};

// y[t][n] (+)= xs[t] * sum_g s[n][g] * sum_{k in g} q[n][k] x[t][k] for n < N,
// t < T.  accumulate: add into y (atomically); otherwise y is overwritten.
int q4_gemm(const uint8_t* packed, int tile0, int N, int ksteps, QAct x, int T, float* y, int ldy, bool accumulate,
            int num_sms, cudaStream_t st);
// The int32 group sums of the same inner loop (T <= 16): out[t][n][g].
int q4_groupsums(const uint8_t* packed, int tile0, int N, int ksteps, QAct x, int T, int32_t* out, cudaStream_t st);

// The head: logits[t][n] = xs[t] * sw[n] * sum_k q[n][k] x[t][k] (int32 sums),
// and, if keys != nullptr, keys[t] = max over n of argmax_key(logits[t][n], n)
// (keys must be zeroed before).
int head_i8(const int8_t* packed, const float* row_scale, int V, int ksteps, QAct x, int T, float* logits, int ldl,
            unsigned long long* keys, int num_sms, cudaStream_t st);

// y[t][n] (+)= sum_k W[n][k] x[t][k]; W f32 [N][K] (K % 4 == 0).
int linear_f32(const float* W, int N, int K, const float* x, int ldx, int T, float* y, int ldy, bool accumulate,
               cudaStream_t st);
// keys[t] = max over n < V of argmax_key(logits[t][n], n).
int argmax_rows(const float* logits, int ldl, int V, int T, unsigned long long* keys, cudaStream_t st);
// tokens[t] = index encoded in keys[t].
int keys_to_tokens(const unsigned long long* keys, int T, uint32_t* tokens, cudaStream_t st);

// ---- layer pieces (k_layer.cu)
// Row maps: output row i reads source row  (i / per) * stride + skip + i % per.
struct RowMap {
    int per, stride, skip;
};
// x = rms(src, w) (w == nullptr: no norm, x = src); then either f32 out
// (out_f32 != nullptr) or int8 codes as f16 + scale (out_q).
int rms_rows(const float* src, int ld_src, RowMap map, int rows, int n, const float* w, float eps, float* out_f32,
             int ld_out, __half* out_codes, float* out_scale, int ld_codes, cudaStream_t st);
// h[r] = embed[tok(r)]: row r of sequence s = r / block_len is the anchor
// (anchor_tok[s]) for r % block_len == 0, the mask token otherwise.
int embed_rows(const float* embed, int H, int vocab, const uint32_t* anchor_tok, int mask_token, int n_seqs,
               int block_len, float* h, cudaStream_t st);
// In-place per-head RMSNorm (q_norm / k_norm) and half-split RoPE of the
// block's q and k: qkv [rows][(nq + 2 nkv) hd]; row r sits at position
// pos0[r / block_len] + r % block_len.
int qk_norm_rope(float* qkv, int ld, int rows, int block_len, const int64_t* pos0_dev, int nq, int nkv, int hd,
                 const float* q_norm, const float* k_norm, const float* inv_freq, float eps, cudaStream_t st);
// Context rows: kv [n][L * 2 * nkv * hd] (per layer k then v) -> the
// sequence's store: K rows normed (k_norm_l) and rotated at position
// pos0 + r, V rows as they are; stored at index (pos0 - first) + r.
int kv_append(const float* kv, int n, int L, int nkv, int hd, const float* const* k_norm_dev, const float* inv_freq,
              float eps, int64_t pos0, int64_t idx0, float* const* kstore_dev, float* const* vstore_dev, int64_t cap,
              cudaStream_t st);
// a = silu(g) * u for gu [rows][2I] (gate then up); f32 out or int8 codes.
int silu_mul(const float* gu, int ld_gu, int rows, int I, float* out_f32, int ld_out, __half* out_codes,
             float* out_scale, int ld_codes, cudaStream_t st);

// Attention of a block over its sequence's context and its own rows.
struct AttnSeq {
    const float* kc;  // layer's key store   [nkv][cap][hd]
    const float* vc;  // layer's value store [nkv][cap][hd]
    int64_t cap;
    int64_t lo;  // first context index read (position - first)
    int n;       // context rows read
};
// qkv [n_seqs*block_len][ld] (q, k, v of the block after norm and RoPE);
// y [n_seqs*block_len][nq*hd].  `part` is scratch of attn_scratch_floats().
int attention(const float* qkv, int ld, int n_seqs, int block_len, const AttnSeq* seqs_dev, int max_ctx, int nq,
              int nkv, int hd, float scale, float* part, int64_t part_floats, float* y, int num_sms, cudaStream_t st);
int64_t attn_scratch_floats(int n_seqs, int block_len, int max_ctx, int nq, int nkv, int hd, int num_sms);

}  // namespace dflash
