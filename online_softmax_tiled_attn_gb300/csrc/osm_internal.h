// osm_internal.h -- declarations shared by the translation units of libosmattn.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "osm_attn.h"

namespace osm {

// Tiled TMA descriptor over a [BH, N, d] bf16 tensor (d innermost): a box of 64 columns x 128
// rows of one (b, h), 128-byte swizzle, zero fill outside [0, N) x [0, d).
int make_bhnd_tensor_map(CUtensorMap* map, const void* base, int64_t BH, int64_t N, int64_t d);

// Tiled TMA descriptor over an explicit mask: uint32 words [Bm, Hm, Nq, W] with the given
// strides in words between heads and sequences (used where Hm, Bm > 1); a box of 4 words
// (one key tile) x 128 query rows, no swizzle, zero fill past Nq.
int make_mask_tensor_map(CUtensorMap* map, const uint32_t* mask, int64_t W, int64_t Nq,
                         int64_t Hm, int64_t Bm, int64_t mask_hs, int64_t mask_bs);

// Deadline of every bounded mbarrier wait in the attention kernel.
unsigned long long fa_wait_timeout_ns();

// Shape of one attention call: Q, O [B, H, Nq, d]; K, V [B, H_kv, Nk, d] (H_kv divides H;
// query head h reads key/value head h / (H / H_kv)); kv_lens, if not null, a device array of
// the B valid key counts (clamped to [0, Nk] in the kernel).  q_pos = 0 means Nq; otherwise
// the rows are packed query heads (see pack_query_heads) with q_pos positions each.
struct AttnShape {
    int64_t B, H, H_kv, Nq, Nk, d;
    const int32_t* kv_lens;
    int64_t q_pos;
    // Optional explicit mask: uint32 words, row i of query head (b, h) at
    // mask + b * mask_bs + h * mask_hs + i * 4 * ceil(Nk / 128); bit j % 32 of word j / 32 set =
    // key j allowed.  Not combined with packed query heads.
    const uint32_t* mask = nullptr;
    int64_t mask_bs = 0, mask_hs = 0;
    // Optional device buffer for the mask's tile map (mask_tile_map_words words): filled by a
    // pre-pass, then key tiles with no allowed key for a whole query tile are skipped.
    uint32_t* tile_map = nullptr;
};

// Words of the tile map of an explicit mask: one row of ceil(ceil(Nk / 128) / 32) words per
// 128-row query tile and mask instance (B instances when mask_bs != 0, times H when
// mask_hs != 0).
int64_t mask_tile_map_words(int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t mask_bs,
                            int64_t mask_hs);

// The same call with the H / H_kv query heads that share a key/value head packed into one row
// block of (H / H_kv) * Nq rows: the [B, H, Nq, d] memory of Q, O and LSE read as
// [B, H_kv, (H / H_kv) * Nq, d].  Each key/value tile is then loaded once per block instead of
// once per query head, and short query blocks (decoding) fill the 128-row tiles.
AttnShape pack_query_heads(const AttnShape& sh);

int fa_fwd_launch(const void* Q, const void* K, const void* V, void* O, float* LSE, int64_t BH,
                  int64_t N, int64_t d, float scale, bool causal, cudaStream_t stream);
int fa_fwd_shape_launch(const void* Q, const void* K, const void* V, void* O, float* LSE,
                        const AttnShape& sh, float scale, bool causal, cudaStream_t stream);
// Number of key ranges the split-key path uses for `requested` (<= 0: chosen from the shape and
// the SM count); 0 when there is no key.
int64_t splitkv_choose_splits(int64_t BH, int64_t Nq, int64_t Nk, int64_t requested);
int fa_fwd_splitkv_launch(const void* Q, const void* K, const void* V, void* O, float* LSE,
                          const AttnShape& sh, float scale, bool causal, int64_t n_splits,
                          float* ws_O, float* ws_LSE, cudaStream_t stream);
int fa_read_device_status(cudaStream_t stream, int* status);
// Device address of the status word the kernels' bounded waits report to (null on failure).
int* device_status_word();
// Q, O, dO, dQ [B, H, N, d]; K, V, dK, dV [B, H_kv, N, d]; LSE, ws_D [B, H, N]; kv_lens null or
// a device int32 [B] of valid keys per sequence.
int fa_bwd_launch(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                  const float* LSE, void* dQ, void* dK, void* dV, float* ws_D, int64_t B,
                  int64_t H, int64_t H_kv, int64_t N, int64_t d, const int32_t* kv_lens,
                  float scale, bool causal, cudaStream_t stream);
int selftest_wait_launch(long long timeout_us, cudaStream_t stream);

int osm_softmax_launch(const float* x, float* y, int64_t rows, int64_t cols, float* lse,
                       cudaStream_t stream);
int osm_softmax_topk_launch(const float* x, int64_t rows, int64_t cols, int64_t k, float* vals,
                            int32_t* idx, float* lse, cudaStream_t stream);

}  // namespace osm
