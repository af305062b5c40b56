// Internal interface of the KV fill paths (generic, decode, tensor core).
#pragma once

#include "common.cuh"

namespace tee {

// Prepared state: header | tensor-core weights | decode-path int4 records (the
// sizes of both fixed by desc and layer count) | RoPE table float2 {cos, sin}
// [max_pos][head_dim/2].
constexpr uint32_t PREP_MAGIC = 0x54454531u;  // "TEE1"
constexpr size_t PREP_HEADER_BYTES = 256;

struct PrepHeader {
    uint32_t magic;
    int32_t d, n_kv_heads, head_dim, max_pos, n_layers, tc_layers, dec_layers;
    int32_t reserved[56];
};
static_assert(sizeof(PrepHeader) == PREP_HEADER_BYTES, "prep header size");

struct FillCall {
    const tee_fill_desc* desc;
    int n_layers;
    const tee_fill_layer* layers;
    const void* prep;
    size_t prep_bytes;
    int n_max;
    const int32_t* n_dev;
    const void* h;
    int64_t ld_h;
    int h_rows;
    const int32_t* rows;
    const int32_t* pos;
    int pos0;
    const int32_t* seq;
    void* k_cache;
    void* v_cache;
    const tee_cache_layout* cache;
    void* ws;
    size_t ws_bytes;
    cudaStream_t stream;
};

struct PrepView {
    const PrepHeader* hdr;  // device pointer
    const char* tc;         // tensor-core weights
    const char* dec;        // decode-path int4 records
    const float2* rope;     // {cos, sin}
};

size_t fill_tc_prep_bytes(const tee_fill_desc& D, int n_layers);
size_t fill_decode_prep_bytes(const tee_fill_desc& D, int n_layers);
inline size_t rope_table_bytes(int max_pos, int hd) {
    return round_up(static_cast<size_t>(max_pos) * (hd / 2) * sizeof(float2), 256);
}
inline PrepView prep_view(const void* prep, const tee_fill_desc& D, int n_layers) {
    PrepView v;
    v.hdr = static_cast<const PrepHeader*>(prep);
    v.tc = static_cast<const char*>(prep) + PREP_HEADER_BYTES;
    v.dec = v.tc + fill_tc_prep_bytes(D, n_layers);
    v.rope = reinterpret_cast<const float2*>(v.dec + fill_decode_prep_bytes(D, n_layers));
    return v;
}

// {cos, sin} of pos * base^(-2i/(2 half)) for pos < max_pos, i < half, computed in float64.
tee_status build_rope_table(float2* table, int max_pos, int half, double base, cudaStream_t s);

// Position check shared by every store: 0 <= p < min(cache max_pos, table length).
__device__ __forceinline__ bool pos_ok(int p, int cache_max, const PrepHeader* hdr) {
    return p >= 0 && p < cache_max && p < hdr->max_pos;
}

__device__ __forceinline__ int item_count(int n_max, const int32_t* n_dev) {
    if (!n_dev) return n_max;
    const int v = *n_dev;
    return v < 0 ? 0 : (v > n_max ? n_max : v);
}

struct GenericWs {
    size_t x_off, r_off, kv_off, end;
};
GenericWs generic_ws(const tee_fill_desc& D, int n_max);

// Tensor-core path (fill_tc.cu): TEE_ERR_UNSUPPORTED when the call does not fit it.
tee_status fill_tc_prepare(const tee_fill_desc& D, int n_layers, const tee_fill_layer* layers, char* tc_area,
                           cudaStream_t s);
size_t fill_tc_ws_bytes(const tee_fill_desc& D, int n_layers, int n_max);
tee_status fill_tc_run(const FillCall& fc);

// Decode path (fill_decode.cu): small item counts; TEE_ERR_UNSUPPORTED otherwise.
// Prepare repacks the int4 weights into the kernel's per-tile block records.
tee_status fill_decode_prepare(const tee_fill_desc& D, int n_layers, const tee_fill_layer* layers, char* area,
                               cudaStream_t s);
size_t fill_decode_ws_bytes(const tee_fill_desc& D, int n_layers, int n_max);
tee_status fill_decode_run(const FillCall& fc);

// Small dense fill (fill_small.cu): the whole chain in one cluster launch for a
// few items on a small model; TEE_ERR_UNSUPPORTED otherwise.
tee_status fill_small_run(const FillCall& fc);

}  // namespace tee
