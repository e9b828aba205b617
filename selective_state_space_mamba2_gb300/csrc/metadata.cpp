// Host-side chunk metadata and slot routing for the varlen SSD prefill.
//
// Follows "[vLLM] Mamba (SSM): 선형 시간 복잡도 시퀀스 모델링", section
// "청크 메타데이터 계산": per request, first close the unaligned remainder of
// the chunk left open by the already-computed tokens, then emit full chunks of
// chunk_size and a partial tail, so that no chunk spans two sequences and a
// state can be stored at every absolute multiple of chunk_size.  Slot routing
// follows "MetadataBuilder 초기화" ("all" mode: one state slot per
// chunk_size block; default mode: one slot per request).
//
// O(S + K) work; pure and deterministic; runs on host memory only.
#include <algorithm>
#include <cstdint>
#include <numeric>
#include <vector>

#include "ssd.h"

extern "C" int32_t ssd_max_chunks(int32_t num_seqs, int32_t total_tokens, int32_t chunk_size) {
    if (num_seqs < 0 || total_tokens < 0 || chunk_size < 1) return -1;
    // a sequence adds at most one partial chunk at each end beyond ceil(T/Q)
    const int64_t bound = 2 * (int64_t)num_seqs + ((int64_t)total_tokens + chunk_size - 1) / chunk_size;
    const int64_t m = bound < total_tokens ? bound : total_tokens;
    return m > INT32_MAX ? INT32_MAX : (int32_t)m;
}

extern "C" ssd_status_t ssd_chunk_metadata(
    int32_t num_seqs, int32_t chunk_size, const int32_t *cu_seqlens,
    const int32_t *num_computed_tokens, const uint8_t *has_initial_states,
    const int32_t *block_table, int64_t block_table_stride, int32_t block_table_cols,
    const int32_t *state_indices, int32_t null_block_id, int32_t max_chunks,
    int32_t *cu_chunk_seqlens, int32_t *seq_idx, int32_t *last_chunk_indices,
    int32_t *chunk_block_col, int32_t *init_slot, int32_t *chunk_slot, int32_t *seq_order,
    int32_t *num_chunks_out) {
    if (num_seqs < 0 || chunk_size < 1 || max_chunks < 0 || !cu_seqlens || !cu_chunk_seqlens ||
        !num_chunks_out || (num_seqs > 0 && (!seq_idx || !last_chunk_indices)))
        return SSD_ERR_INVALID_ARG;
    if (cu_seqlens[0] != 0) return SSD_ERR_INVALID_ARG;
    if (block_table && (block_table_cols < 1 || block_table_stride < block_table_cols))
        return SSD_ERR_INVALID_ARG;

    int32_t k = 0;  // chunks emitted so far
    auto emit = [&](int32_t end_token, int32_t r, int64_t abs_last_pos) -> bool {
        if (k >= max_chunks) return false;
        cu_chunk_seqlens[k + 1] = end_token;
        seq_idx[k] = r;
        const int32_t col = (int32_t)(abs_last_pos / chunk_size);
        if (chunk_block_col) chunk_block_col[k] = col;
        ++k;
        return true;
    };
    cu_chunk_seqlens[0] = 0;

    for (int32_t r = 0; r < num_seqs; ++r) {
        const int32_t start = cu_seqlens[r];
        const int32_t end = cu_seqlens[r + 1];
        if (end < start) return SSD_ERR_INVALID_ARG;
        const int64_t computed = num_computed_tokens ? num_computed_tokens[r] : 0;
        if (computed < 0) return SSD_ERR_INVALID_ARG;
        const bool has_init = has_initial_states && has_initial_states[r];

        if (init_slot) {
            int32_t slot = null_block_id;
            if (has_init) {
                if (block_table) {
                    if (computed == 0) return SSD_ERR_INVALID_ARG;
                    const int64_t col = (computed - 1) / chunk_size;
                    if (col >= block_table_cols) return SSD_ERR_INVALID_ARG;
                    slot = block_table[(int64_t)r * block_table_stride + col];
                } else if (state_indices) {
                    slot = state_indices[r];
                }
            }
            init_slot[r] = slot;
        }

        const int32_t first_chunk = k;
        int32_t pos_tok = start;       // next packed token to place
        int64_t abs_pos = computed;    // its absolute position in the request
        int32_t remaining = end - start;
        // 1. close the partially filled chunk left by the computed prefix
        if (remaining > 0 && abs_pos % chunk_size != 0) {
            int64_t len = (abs_pos / chunk_size + 1) * chunk_size - abs_pos;
            if (len > remaining) len = remaining;
            pos_tok += (int32_t)len;
            abs_pos += len;
            remaining -= (int32_t)len;
            if (!emit(pos_tok, r, abs_pos - 1)) return SSD_ERR_WORKSPACE;
        }
        // 2. full chunks, then the partial tail
        while (remaining > 0) {
            const int32_t len = remaining < chunk_size ? remaining : chunk_size;
            pos_tok += len;
            abs_pos += len;
            remaining -= len;
            if (!emit(pos_tok, r, abs_pos - 1)) return SSD_ERR_WORKSPACE;
        }
        last_chunk_indices[r] = k - 1;

        if (chunk_slot) {
            for (int32_t c = first_chunk; c < k; ++c) {
                int32_t slot = null_block_id;
                if (block_table) {
                    const int64_t col = (int64_t)(computed + (cu_chunk_seqlens[c + 1] - 1 - start)) / chunk_size;
                    if (col >= block_table_cols) return SSD_ERR_INVALID_ARG;
                    slot = block_table[(int64_t)r * block_table_stride + col];
                } else if (state_indices && c == k - 1) {
                    slot = state_indices[r];
                }
                chunk_slot[c] = slot;
            }
        }
    }
    if (seq_order) {
        std::vector<int32_t> idx(num_seqs);
        std::iota(idx.begin(), idx.end(), 0);
        std::stable_sort(idx.begin(), idx.end(), [&](int32_t a, int32_t b) {
            return cu_seqlens[a + 1] - cu_seqlens[a] > cu_seqlens[b + 1] - cu_seqlens[b];
        });
        std::copy(idx.begin(), idx.end(), seq_order);
    }
    *num_chunks_out = k;
    return SSD_OK;
}
