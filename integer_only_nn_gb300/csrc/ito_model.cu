// The model: a sequential stack of trainable int8 layers and the whole NITI
// training step ("Integer On-Device Training: Overview", section 4:
// INT_LAYERS[] of layer descriptors with mutable int8 weights, the training
// loop INTODT_Forward -> compute_loss -> INTODT_Backward; section 3 for the
// arithmetic; section 9, "Trained Weights in RAM", for the checkpoint).
//
// Layout in device memory (allocated once at creation):
//   per layer l: W8 [OC][K] int8 (the weights) and Wb, its bf16 copy that the
//   tensor cores read (row pitch rounded up to 8 elements); y32 [rows][OC]
//   int32 forward contraction; a8 [rows][OC] int8 output (+ bf16 copy when a
//   Linear layer reads it); e8/eb the delta at the layer output; d32 the int32
//   delta-propagation contraction at the layer input; g32 [OC][K] int32
//   weight gradient; for conv layers Pb, the bf16 im2col patches of the layer
//   input, and dcol, the int32 patch-space delta.
//   stats: int32 scalars, 8 per layer (ymax, ys, dmax, ds, gmax, gs, ws, nz)
//   then pmax, ps of the pooling layer.
// Step order: forward over all layers; top error; for each layer from the top
// down: delta propagation with the weights before this step's update (not for
// the first layer), weight gradient, NITI update.
#include <algorithm>
#include <cstdlib>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "ito_conv.h"
#include "ito_device.cuh"
#include "ito_internal.h"

namespace ito {

enum {
    ST_YMAX = 0, ST_YS, ST_DMAX, ST_DS, ST_GMAX, ST_GS, ST_WS, ST_NZ,
    ST_OGMAX, ST_OGS, ST_OWS, ST_ONZ,   // offsets of a statically requantised layer
    ST_PER_LAYER
};

struct MLayer {
    int kind;
    int IC, OC;
    int H, W, OH, OW, stride;   // conv
    int64_t K;                  // forward contraction length (IC or 9*IC)
    int64_t rows_in, rows_out;  // B or B*H*W / B*OH*OW
    int8_t* W8 = nullptr;
    uint16_t* Wb = nullptr;
    int64_t ldw = 0;
    uint16_t* Pb = nullptr;     // conv patches [rows_out][ldp]
    int64_t ldp = 0;
    int32_t* y32 = nullptr;
    int8_t* a8 = nullptr;
    uint16_t* ab = nullptr;     // bf16 copy of the output (read by a following Linear)
    int64_t lda = 0;
    int8_t* e8 = nullptr;       // delta at the output
    uint16_t* eb = nullptr;
    int64_t lde = 0;
    int32_t* dcol = nullptr;    // conv: [rows_out][K]
    int32_t* d32 = nullptr;     // [rows_in][IC]
    int32_t* g32 = nullptr;     // [OC][K]
    uint8_t* mask = nullptr;    // bit-packed ReLU mask of the output [rows][OC / 8] (packed_masks)
    bool static_q = false;      // static per-channel requantisation with trained INT32 offsets
    int32_t *off32 = nullptr, *mult32 = nullptr, *k32 = nullptr, *og32 = nullptr;   // [OC] (Linear layers)
    GemmPlan pf{}, pd{}, pg{};
    // speculative requantisation (see FusedRq): pf / pd with the requantising epilogue, and their
    // re-launches, which check the shift prediction and recompute when it missed
    GemmPlan pf_spec{}, pd_spec{}, pf_redo{}, pd_redo{};
    // stride-2 conv: the input-space delta by parity phases (no patch-space delta, no gather)
    bool s2 = false;
    ConvS2Plan ps2{};
    // stride-2 conv after a conv: forward and weight gradient on the parity planes of the
    // previous layer's bf16 output copy (no im2col patches)
    bool ig = false;
    ConvIgPlan pig_f{}, pig_g{};
    bool has_dgrad = false;
    bool relu = false;
};

}  // namespace ito

struct ito_model {
    int batch = 0;
    ito_niti_params p{};
    ito_model_options opt{};
    int32_t target_mag = 64;
    int n_conv = 0;
    bool has_pool = false;
    int pool_C = 0, pool_HW = 0;
    int in_features = 0;         // elements per sample of the input
    std::vector<ito::MLayer> L;
    // input
    int8_t* x8 = nullptr;        // model-owned input (host-path steps)
    int32_t* labels = nullptr;
    // pipelined host-path steps: a second input buffer pair, the copy stream, and per buffer
    // "copied" / "read by its step" events
    int8_t* x8b = nullptr;
    int32_t* labels_b = nullptr;
    cudaStream_t copy_stream = nullptr;
    cudaEvent_t ev_copied[2] = {nullptr, nullptr}, ev_consumed[2] = {nullptr, nullptr};
    int64_t async_steps = 0;
    uint16_t* xb = nullptr;      // bf16 copy of a Linear first layer's input
    int64_t ldx = 0;
    // pooling
    int32_t* p32 = nullptr;
    int8_t* pa8 = nullptr;
    uint16_t* pab = nullptr;
    int8_t* pe8 = nullptr;
    // ping-pong delta buffers (pingpong_grads)
    int8_t* gbuf8[2] = {nullptr, nullptr};
    uint16_t* gbufb[2] = {nullptr, nullptr};
    int32_t* stats = nullptr;
    int n_stats = 0;
    uint32_t* discard_max = nullptr;   // max target of the patch-space conv delta (not a NITI tensor)
    int32_t* split_ws = nullptr;       // split-K partials, shared by the step's contractions (one stream)
    size_t split_ws_bytes = 0;
    int32_t* split_ws_g = nullptr;     // the weight gradients' own (they may run beside the others, mode 3)
    std::vector<void*> allocs;
    std::vector<std::pair<std::string, int>> stat_names;
    // CUDA-graph replay of whole steps, keyed by the caller's input pointers
    struct GraphEntry {
        const void* x;
        const void* labels;
        cudaGraphExec_t exec;
        int launches;
        std::vector<int> prof_cls;       // event pairs captured into the graph (profiling on)
        std::vector<double> prof_work;
    };
    bool graph_on = false;
    bool graph_warm = false;
    bool capturing = false;      // a step is being captured into a graph
    std::vector<GraphEntry> graphs;
    // backward overlap: the bandwidth passes (requantisation of the propagated delta, the
    // weight and offset updates) run on a second stream beside the next contractions
    int overlap = 1;                    // 0: one stream; 1: requantisation and updates overlap; 2: updates only;
                                        // 3: weight gradients and updates beside the delta chain
    bool overlap3_ok = false;           // mode 3 is possible (no ping-pong buffers, no static requantisation)
    // speculative requantisation: [0, nl) forward and [nl, 2nl) delta-propagation shift predictions,
    // then the shifts of the last step in the same order, then 1 where the contraction's epilogue
    // speculates (its plan is fused), then the re-launch words (0: the prediction held, else the
    // shift + 1); spec_count: predictions that held, that missed (int64)
    bool speculate = true;
    int32_t* spec = nullptr;
    int64_t* spec_count = nullptr;
    int32_t* pred_y(int l) { return spec + l; }
    int32_t* pred_d(int l) { return spec + (int)L.size() + l; }
    int32_t* last_y(int l) { return spec + 2 * (int)L.size() + l; }
    int32_t* last_d(int l) { return spec + 3 * (int)L.size() + l; }
    int32_t* redo_y(int l) { return spec + 6 * (int)L.size() + l; }
    int32_t* redo_d(int l) { return spec + 7 * (int)L.size() + l; }
    cudaStream_t side = nullptr;
    // [0] fork, [1] join, then per layer: propagated delta computed, requantised delta ready,
    // weight gradient computed
    std::vector<cudaEvent_t> sync_ev;
    cudaEvent_t ev_fork() const { return sync_ev[0]; }
    cudaEvent_t ev_join() const { return sync_ev[1]; }
    cudaEvent_t ev_dgrad(int l) const { return sync_ev[2 + 3 * l]; }
    cudaEvent_t ev_delta(int l) const { return sync_ev[3 + 3 * l]; }
    cudaEvent_t ev_wgrad(int l) const { return sync_ev[4 + 3 * l]; }
    // measurement hooks
    bool prof_on = false;
    std::vector<cudaEvent_t> prof_ev;      // pairs (begin, end)
    std::vector<int> prof_cls;
    std::vector<double> prof_work;
    int prof_n = 0;
    int launches = 0;                      // kernels launched by the current / last step
    bool top_fused = false;                // this step's forward wrote the top error

    // during a capture the record must be "external" to become a graph node (the flag is
    // rejected on a stream that is not capturing)
    void record(cudaEvent_t e, cudaStream_t s)
    {
        if (capturing)
            cudaEventRecordWithFlags(e, s, cudaEventRecordExternal);
        else
            cudaEventRecord(e, s);
    }
    void grow_events(size_t n)
    {
        while (prof_ev.size() < n) {
            cudaEvent_t e;
            cudaEventCreate(&e);
            prof_ev.push_back(e);
        }
    }
    void mark_begin(cudaStream_t s)
    {
        ++launches;
        if (!prof_on) return;
        if ((size_t)(2 * prof_n + 2) > prof_ev.size()) grow_events(prof_ev.size() + 128);
        record(prof_ev[2 * prof_n], s);
    }
    void mark_end(cudaStream_t s, int cls, double work)
    {
        if (!prof_on) return;
        record(prof_ev[2 * prof_n + 1], s);
        prof_cls.push_back(cls);
        prof_work.push_back(work);
        ++prof_n;
    }

    template <class T>
    int alloc(T** out, size_t count)
    {
        void* p = nullptr;
        if (count == 0) count = 1;
        cudaError_t e = cudaMalloc(&p, count * sizeof(T));
        if (e != cudaSuccess) return ito::set_error(ITO_ERR_CUDA, "cudaMalloc: %s", cudaGetErrorString(e));
        cudaMemset(p, 0, count * sizeof(T));
        allocs.push_back(p);
        *out = static_cast<T*>(p);
        return ITO_OK;
    }
    uint32_t* umax(int l, int which) { return reinterpret_cast<uint32_t*>(stats + l * ito::ST_PER_LAYER + which); }
    int32_t* sval(int l, int which) { return stats + l * ito::ST_PER_LAYER + which; }
};

using namespace ito;

#define ITO_TRY(x)                   \
    do {                             \
        int _r = (x);                \
        if (_r != ITO_OK) return _r; \
    } while (0)

static int build_model(ito_model* m, const ito_layer_desc* d, int n)
{
    const int B = m->batch;
    // parse: conv* [gap] linear* (last one ITO_LAYER_LINEAR)
    int i = 0;
    while (i < n && d[i].kind == ITO_LAYER_CONV3X3_RELU) ++i;
    m->n_conv = i;
    if (i < n && d[i].kind == ITO_LAYER_GAP) {
        m->has_pool = true;
        ++i;
    }
    const int first_linear = i;
    for (; i < n; ++i) {
        if (d[i].kind != ITO_LAYER_LINEAR_RELU && d[i].kind != ITO_LAYER_LINEAR)
            return set_error(ITO_ERR_UNSUPPORTED, "layer %d: order must be conv*, [gap], linear*", i);
        if (d[i].kind == ITO_LAYER_LINEAR && i != n - 1)
            return set_error(ITO_ERR_UNSUPPORTED, "only the last layer may be a plain Linear");
    }
    if (first_linear >= n || d[n - 1].kind != ITO_LAYER_LINEAR)
        return set_error(ITO_ERR_UNSUPPORTED, "the stack must end with one ITO_LAYER_LINEAR");
    if (m->n_conv > 0 && !m->has_pool) return set_error(ITO_ERR_UNSUPPORTED, "conv layers must be followed by GAP");

    // shapes
    int H = 0, W = 0, C = 0;
    if (m->n_conv > 0) {
        H = d[0].in_h;
        W = d[0].in_w;
        C = d[0].in_features;
        if (H < 1 || W < 1 || C < 1) return set_error(ITO_ERR_SHAPE, "conv input size");
        m->in_features = H * W * C;
    } else {
        m->in_features = d[first_linear].in_features;
    }
    for (int l = 0; l < m->n_conv; ++l) {
        const ito_layer_desc& q = d[l];
        if (q.in_features != C || q.in_h != H || q.in_w != W) return set_error(ITO_ERR_SHAPE, "conv %d input", l);
        if (q.stride != 1 && q.stride != 2) return set_error(ITO_ERR_SHAPE, "conv %d stride", l);
        if (q.out_features < 1 || q.out_features % 8 || (l > 0 && C % 8))
            return set_error(ITO_ERR_UNSUPPORTED, "conv %d channels must be multiples of 8", l);
        MLayer L;
        L.kind = q.kind;
        L.IC = C;
        L.OC = q.out_features;
        L.H = H;
        L.W = W;
        L.stride = q.stride;
        L.OH = (H + 2 - 3) / q.stride + 1;
        L.OW = (W + 2 - 3) / q.stride + 1;
        L.K = 9LL * C;
        L.rows_in = (int64_t)B * H * W;
        L.rows_out = (int64_t)B * L.OH * L.OW;
        L.relu = true;
        L.has_dgrad = l > m->opt.trainable_from;
        m->L.push_back(L);
        H = L.OH;
        W = L.OW;
        C = L.OC;
    }
    int F;
    if (m->has_pool) {
        const ito_layer_desc& q = d[m->n_conv];
        if (m->n_conv == 0) return set_error(ITO_ERR_UNSUPPORTED, "GAP needs conv layers before it");
        if (q.in_features != C) return set_error(ITO_ERR_SHAPE, "GAP channels");
        m->pool_C = C;
        m->pool_HW = H * W;
        F = C;
    } else {
        F = m->in_features;
    }
    for (int l = first_linear; l < n; ++l) {
        const ito_layer_desc& q = d[l];
        if (q.in_features != F || q.out_features < 1) return set_error(ITO_ERR_SHAPE, "linear %d features", l);
        MLayer L;
        L.kind = q.kind;
        L.IC = F;
        L.OC = q.out_features;
        L.H = L.W = L.OH = L.OW = 1;
        L.stride = 0;
        L.K = F;
        L.rows_in = L.rows_out = B;
        L.relu = q.kind == ITO_LAYER_LINEAR_RELU;
        L.has_dgrad = (int)m->L.size() > m->opt.trainable_from;
        m->L.push_back(L);
        F = q.out_features;
    }
    const int nl = (int)m->L.size();
    if (m->opt.trainable_from < 0 || m->opt.trainable_from >= nl)
        return set_error(ITO_ERR_ARG, "trainable_from must be in [0, %d)", nl);
    if (m->opt.input_uint8 && m->n_conv > 0)
        return set_error(ITO_ERR_UNSUPPORTED, "UINT8 input is supported for a Linear first layer");
    if (m->opt.packed_masks)
        for (int l = 0; l < nl; ++l)
            if (m->L[l].relu && m->L[l].OC % 8)
                return set_error(ITO_ERR_UNSUPPORTED, "packed masks need ReLU widths that are multiples of 8");

    for (int l = 1; l < nl; ++l) {
        MLayer& L = m->L[l];
        L.ig = L.kind == ITO_LAYER_CONV3X3_RELU && m->L[l - 1].kind == ITO_LAYER_CONV3X3_RELU &&
               conv_dgrad_s2_eligible(B, L.H, L.W, L.IC, L.OC, L.stride);
    }

    // allocations
    ITO_TRY(m->alloc(&m->x8, (size_t)B * m->in_features));
    ITO_TRY(m->alloc(&m->labels, (size_t)B));
    ITO_TRY(m->alloc(&m->x8b, (size_t)B * m->in_features));
    ITO_TRY(m->alloc(&m->labels_b, (size_t)B));
    m->n_stats = nl * ST_PER_LAYER + 2;
    ITO_TRY(m->alloc(&m->stats, (size_t)m->n_stats));
    ITO_TRY(m->alloc(&m->discard_max, 1));
    if (m->n_conv == 0) {
        m->ldx = pad8(m->in_features);
        ITO_TRY(m->alloc(&m->xb, (size_t)B * m->ldx));
    }
    if (m->has_pool) {
        ITO_TRY(m->alloc(&m->p32, (size_t)B * m->pool_C));
        ITO_TRY(m->alloc(&m->pa8, (size_t)B * m->pool_C));
        ITO_TRY(m->alloc(&m->pab, (size_t)B * pad8(m->pool_C)));
        ITO_TRY(m->alloc(&m->pe8, (size_t)B * m->pool_C));
    }
    for (int l = 0; l < nl; ++l) {
        MLayer& L = m->L[l];
        const bool conv = L.kind == ITO_LAYER_CONV3X3_RELU;
        L.ldw = pad8(L.K);
        ITO_TRY(m->alloc(&L.W8, (size_t)L.OC * L.K));
        ITO_TRY(m->alloc(&L.Wb, (size_t)L.OC * L.ldw));
        ITO_TRY(m->alloc(&L.y32, (size_t)L.rows_out * L.OC));
        ITO_TRY(m->alloc(&L.a8, (size_t)L.rows_out * L.OC));
        L.lda = pad8(L.OC);
        const bool next_linear = l + 1 < nl && m->L[l + 1].kind != ITO_LAYER_CONV3X3_RELU && !conv;
        const bool next_planes = l + 1 < nl && m->L[l + 1].ig;   // the next conv reads this output's bf16 copy
        if (next_linear || next_planes) ITO_TRY(m->alloc(&L.ab, (size_t)L.rows_out * L.lda));
        L.lde = pad8(L.OC);
        if (m->opt.pingpong_grads) {
            // two delta buffers for all layers: layer l writes buffer l % 2, which no layer
            // still needs (layer l + 2's delta was consumed by its weight gradient and update)
            if (!m->gbuf8[0]) {
                size_t n8 = 0, nb = 0;
                for (const MLayer& Q : m->L) {
                    n8 = std::max(n8, (size_t)Q.rows_out * Q.OC);
                    nb = std::max(nb, (size_t)Q.rows_out * pad8(Q.OC));
                }
                for (int i = 0; i < 2; ++i) {
                    ITO_TRY(m->alloc(&m->gbuf8[i], n8));
                    ITO_TRY(m->alloc(&m->gbufb[i], nb));
                }
            }
            L.e8 = m->gbuf8[l % 2];
            L.eb = m->gbufb[l % 2];
        } else {
            ITO_TRY(m->alloc(&L.e8, (size_t)L.rows_out * L.OC));
            ITO_TRY(m->alloc(&L.eb, (size_t)L.rows_out * L.lde));
        }
        ITO_TRY(m->alloc(&L.g32, (size_t)L.OC * L.K));
        if (m->opt.packed_masks && L.relu) ITO_TRY(m->alloc(&L.mask, (size_t)L.rows_out * (L.OC / 8)));
        if (!conv) {
            ITO_TRY(m->alloc(&L.off32, (size_t)L.OC));
            ITO_TRY(m->alloc(&L.mult32, (size_t)L.OC));
            ITO_TRY(m->alloc(&L.k32, (size_t)L.OC));
            ITO_TRY(m->alloc(&L.og32, (size_t)L.OC));
        }
        if (L.has_dgrad) ITO_TRY(m->alloc(&L.d32, (size_t)L.rows_in * L.IC));
        if (conv) {
            L.ldp = pad8(L.K);
            if (!L.ig) ITO_TRY(m->alloc(&L.Pb, (size_t)L.rows_out * L.ldp));
            L.s2 = L.has_dgrad && conv_dgrad_s2_eligible(B, L.H, L.W, L.IC, L.OC, L.stride);
            if (L.has_dgrad && !L.s2) ITO_TRY(m->alloc(&L.dcol, (size_t)L.rows_out * L.K));
        }
    }

    // split-K partials: one buffer for the largest need (the step's kernels run in order)
    for (int l = 0; l < nl; ++l) {
        const MLayer& L = m->L[l];
        const int M = (int)L.rows_out;
        size_t need = gemm_split_ws_bytes(M, L.OC, (int)L.K, L.OC);
        if (L.has_dgrad) need = std::max(need, gemm_split_ws_bytes(M, (int)L.K, L.OC, L.K));
        need = std::max(need, gemm_split_ws_bytes(L.OC, (int)L.K, M, L.K));
        if (L.ig) need = std::max(need, conv_wgrad_s2_ws_bytes(B, L.H, L.W, L.IC, L.OC));
        m->split_ws_bytes = std::max(m->split_ws_bytes, need);
    }
    if (m->split_ws_bytes) ITO_TRY(m->alloc(&m->split_ws, m->split_ws_bytes / sizeof(int32_t)));
    // mode 3 runs each weight gradient beside the next delta propagation: their partials
    // get their own workspace, and the delta buffers must not be shared
    m->overlap3_ok = !m->opt.pingpong_grads;
    for (const MLayer& L : m->L)
        if (L.static_q) m->overlap3_ok = false;
    if (m->overlap3_ok && m->split_ws_bytes)
        ITO_TRY(m->alloc(&m->split_ws_g, m->split_ws_bytes / sizeof(int32_t)));
    int32_t* const ws_g = m->overlap3_ok ? m->split_ws_g : m->split_ws;
    ITO_TRY(m->alloc(&m->spec, (size_t)8 * nl));
    ITO_TRY(m->alloc(&m->spec_count, 2));
    if (cudaMemset(m->spec, 0xff, sizeof(int32_t) * 4 * nl) != cudaSuccess)   // -1: no prediction yet
        return set_error(ITO_ERR_CUDA, "memset");
    m->speculate = true;   // ito_model_set_speculation turns it off

    // contraction plans (tensor maps over the buffers above)
    for (int l = 0; l < nl; ++l) {
        MLayer& L = m->L[l];
        const bool conv = L.kind == ITO_LAYER_CONV3X3_RELU;
        uint32_t* ymax = m->umax(l, ST_YMAX);
        uint32_t* dmax = m->umax(l, ST_DMAX);
        uint32_t* gmax = m->umax(l, ST_GMAX);
        const Bf16View wv{L.Wb, L.OC, L.K, L.ldw};
        const Bf16View ev{L.eb, L.rows_out, L.OC, L.lde};
        Bf16View in;
        if (conv) {
            in = Bf16View{L.Pb, L.rows_out, L.K, L.ldp};
        } else if (l == m->n_conv && m->has_pool) {
            in = Bf16View{m->pab, B, L.IC, pad8(L.IC)};
        } else if (l == 0) {
            in = Bf16View{m->xb, B, L.IC, m->ldx};
        } else {
            in = Bf16View{m->L[l - 1].ab, B, L.IC, m->L[l - 1].lda};
        }
        const int M = (int)L.rows_out;
        // a UINT8 input makes products up to 255 * 128: shorter exact chunks
        const int chunk = (l == 0 && m->opt.input_uint8) ? kExactChunkU8 : kExactChunk;
        // The CTA-pair kernel only for contractions of at least 64 pair tiles: on fewer the
        // single-CTA kernel is faster (784-1024x3-10 MLP, batch 256: 0.142 against 0.153 ms
        // per step; the CNN 0.385 against 0.395 ms). A model that asks for speculative
        // requantisation below its default size gets the pair kernel there (the requantising
        // epilogue is the pair kernel's).
        const int64_t spec_min = m->opt.speculate_min_elems > 0 ? m->opt.speculate_min_elems : (int64_t)1 << 22;
        const bool spec_small = m->opt.speculate_min_elems > 0;
        constexpr int kMinPairTiles = 64;
        const int pair_f = spec_small && L.rows_out * L.OC >= spec_min ? 1 : kMinPairTiles;
        const int pair_d = spec_small && L.rows_in * L.IC >= spec_min ? 1 : kMinPairTiles;
        if (L.ig) {
            // forward and weight gradient on the parity planes of the previous conv's bf16 output
            const MLayer& prev = m->L[l - 1];
            ITO_TRY(conv_fwd_s2_plan(&L.pig_f, prev.ab, prev.lda, L.Wb, L.ldw, B, L.H, L.W, L.IC, L.OC, L.y32, ymax));
            ITO_TRY(conv_wgrad_s2_plan(&L.pig_g, L.eb, L.lde, prev.ab, prev.lda, B, L.H, L.W, L.IC, L.OC, L.g32, gmax,
                                       ws_g, m->split_ws_bytes));
        } else {
            // forward: Y[m][oc] = sum_k in[m][k] W[oc][k]
            ITO_TRY(gemm_plan(&L.pf, in, false, wv, false, M, L.OC, (int)L.K, L.y32, L.OC, ymax, m->split_ws,
                              m->split_ws_bytes, chunk, pair_f));
        }
        // delta propagation: D[m][k] = sum_oc e[m][oc] W[oc][k]; for a conv this is the
        // patch-space delta, whose max is not the NITI max (col2im takes that), except for a
        // stride-2 conv, whose input-space delta comes straight from its parity phases
        if (L.s2)
            ITO_TRY(conv_dgrad_s2_plan(&L.ps2, L.eb, L.lde, L.Wb, L.ldw, B, L.H, L.W, L.IC, L.OC, L.d32, dmax));
        else if (L.has_dgrad)
            ITO_TRY(gemm_plan(&L.pd, ev, false, wv, true, M, (int)L.K, L.OC, conv ? L.dcol : L.d32, L.K,
                              conv ? m->discard_max : dmax, m->split_ws, m->split_ws_bytes, kExactChunk, pair_d));
        // weight gradient: G[oc][k] = sum_m e[m][oc] in[m][k]
        if (!L.ig)
            ITO_TRY(gemm_plan(&L.pg, ev, true, in, true, L.OC, (int)L.K, M, L.g32, L.K, gmax, ws_g,
                              m->split_ws_bytes, chunk, kMinPairTiles));
        // speculative requantisation in the epilogues of the forward contraction (its ReLU'd
        // activation and bf16 copy) and of the delta propagation (the gated delta below); not
        // with bit-packed masks, static requantisation, or shared (ping-pong) delta buffers
        const bool plain = !m->opt.packed_masks && !m->opt.pingpong_grads;
        L.pf_spec = L.pf;
        L.pd_spec = L.pd;
        if (plain && !conv && !L.static_q && L.ab && L.rows_out * L.OC >= spec_min)
            ITO_TRY(gemm_plan_fuse_requant(&L.pf_spec, m->pred_y(l), L.relu ? 1 : 0, nullptr, 0, L.a8, L.OC, L.ab,
                                           L.lda));
        if (plain && !conv && L.has_dgrad && !(l == m->n_conv && m->has_pool) && L.rows_in * L.IC >= spec_min) {
            const MLayer& prev = m->L[l - 1];
            if (prev.kind != ITO_LAYER_CONV3X3_RELU)
                ITO_TRY(gemm_plan_fuse_requant(&L.pd_spec, m->pred_d(l), 0, prev.relu ? prev.a8 : nullptr, L.IC,
                                               prev.e8, L.IC, prev.eb, prev.lde));
        }
        // the re-launches: the same plans, with the check of the prediction in their prologue
        if (L.pf_spec.rq_pred) {
            L.pf_redo = L.pf_spec;
            L.pf_redo.rq_redo = m->redo_y(l);
            L.pf_redo.rq_d_shift = m->sval(l, ST_YS);
            L.pf_redo.rq_s_last = m->last_y(l);
            L.pf_redo.rq_target_bits = m->p.target_bits;
        }
        if (L.pd_spec.rq_pred) {
            L.pd_redo = L.pd_spec;
            L.pd_redo.rq_redo = m->redo_d(l);
            L.pd_redo.rq_d_shift = m->sval(l, ST_DS);
            L.pd_redo.rq_s_last = m->last_d(l);
            L.pd_redo.rq_target_bits = m->p.target_bits;
        }
    }
    {
        // the slots whose contraction plan took the fused epilogue (a plan may decline it)
        std::vector<int32_t> used(2 * nl, 0);
        for (int l = 0; l < nl; ++l) {
            used[l] = m->L[l].pf_spec.rq_pred != nullptr;
            used[nl + l] = m->L[l].pd_spec.rq_pred != nullptr;
        }
        if (cudaMemcpy(m->spec + 4 * nl, used.data(), sizeof(int32_t) * 2 * nl, cudaMemcpyHostToDevice) !=
            cudaSuccess)
            return set_error(ITO_ERR_CUDA, "memcpy");
    }

    // names of the stats entries
    const char* nm[ST_PER_LAYER] = {"ymax", "ys", "dmax", "ds", "gmax", "gs", "ws", "nz",
                                    "ogmax", "ogs", "ows", "onz"};
    for (int l = 0; l < nl; ++l)
        for (int k = 0; k < ST_PER_LAYER; ++k) m->stat_names.push_back({std::string(nm[k]) + std::to_string(l),
                                                                         l * ST_PER_LAYER + k});
    m->stat_names.push_back({"pmax", nl * ST_PER_LAYER});
    m->stat_names.push_back({"ps", nl * ST_PER_LAYER + 1});

    // second stream and ordering events of the backward overlap: mode 1 unless every delta
    // propagation speculates; then the second stream would hold only the weight updates,
    // which slow the contractions beside them by more than they take alone, so it takes the
    // weight gradients too (mode 3: they fill the partial last waves of the delta
    // propagations; batch-8192 MLP 1.996 -> 1.976 ms a step), or nothing (mode 0) where mode 3
    // is not possible (ito_model_set_overlap changes it)
    {
        bool every_delta_speculates = m->speculate;
        for (const MLayer& L : m->L)
            if (L.has_dgrad && !L.pd_spec.rq_pred) every_delta_speculates = false;
        m->overlap = every_delta_speculates ? (m->overlap3_ok ? 3 : 0) : 1;
    }
    if (cudaStreamCreateWithFlags(&m->side, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&m->copy_stream, cudaStreamNonBlocking) != cudaSuccess)
        return set_error(ITO_ERR_CUDA, "stream creation failed");
    for (int i = 0; i < 2; ++i)
        if (cudaEventCreateWithFlags(&m->ev_copied[i], cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&m->ev_consumed[i], cudaEventDisableTiming) != cudaSuccess)
            return set_error(ITO_ERR_CUDA, "event creation failed");
    for (int i = 0; i < 2 + 3 * nl; ++i) {
        cudaEvent_t e;
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess)
            return set_error(ITO_ERR_CUDA, "event creation failed");
        m->sync_ev.push_back(e);
    }
    return cudaDeviceSynchronize() == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "model init sync");
}

// Launch `call` bracketed by the model's measurement marks.
#define ITO_LAUNCH(m, s, cls, work, call)      \
    do {                                       \
        (m)->mark_begin(s);                    \
        int _r = (call);                       \
        (m)->mark_end(s, cls, (double)(work)); \
        if (_r != ITO_OK) return _r;           \
    } while (0)

static double gemm_ops(const GemmPlan& g) { return 2.0 * g.M * (double)g.N * g.K; }

// algorithmic HBM bytes of a requantisation pass: int32 in, int8 out, bf16 copy, gate
static double requant_bytes(int64_t n, bool bf16, bool gate)
{
    return (double)n * (4 + 1 + (bf16 ? 2 : 0) + (gate ? 1 : 0));
}

// The start of a step: statistics zeroed, shift predictions rolled (a training step), and a
// Linear first layer's input converted to its bf16 copy, in one launch.
static int model_begin(ito_model* m, const int8_t* x, bool train, cudaStream_t s)
{
    const int B = m->batch;
    const int nl = (int)m->L.size();
    const bool conv_in = m->n_conv > 0;
    ITO_LAUNCH(m, s, ITO_PROF_OTHER, conv_in ? 4.0 * m->n_stats : 3.0 * B * m->in_features + 4.0 * m->n_stats,
               launch_step_begin(m->stats, m->n_stats, m->spec, m->spec + 2 * nl, m->spec + 4 * nl, m->spec_count,
                                 train ? 2 * nl : 0, m->speculate ? 1 : 0, conv_in ? nullptr : x,
                                 m->opt.input_uint8 ? 1 : 0, B, m->in_features, m->xb, m->ldx, s));
    return ITO_OK;
}

// labels: the step's labels (the top error is computed beside the logits' requantisation),
// or nullptr (inference)
static int model_forward(ito_model* m, const int8_t* x, const int32_t* labels, cudaStream_t s)
{
    const int B = m->batch;
    const int nl = (int)m->L.size();
    const ito_niti_params p = m->p;
    m->top_fused = false;
    const int8_t* in8 = x;
    for (int l = 0; l < nl; ++l) {
        MLayer& L = m->L[l];
        if (L.kind == ITO_LAYER_CONV3X3_RELU && !L.ig) {
            ITO_LAUNCH(m, s, ITO_PROF_OTHER, (double)L.rows_in * L.IC + 2.0 * L.rows_out * L.ldp,
                       launch_im2col(in8, B, L.H, L.W, L.IC, L.OH, L.OW, L.stride, L.Pb, L.ldp, s));
        } else if (l == m->n_conv && m->has_pool) {
            const int pl = nl;   // pooling scalars follow the per-layer block
            uint32_t* pmax = reinterpret_cast<uint32_t*>(m->stats + pl * ST_PER_LAYER);
            ITO_LAUNCH(m, s, ITO_PROF_OTHER, (double)B * m->pool_C * (m->pool_HW + 4),
                       launch_gap_fwd(in8, B, m->pool_HW, m->pool_C, m->p32, pmax, s));
            ITO_LAUNCH(m, s, ITO_PROF_REQUANT, requant_bytes((int64_t)B * m->pool_C, true, false),
                       launch_requant(m->p32, B, m->pool_C, pmax, p.target_bits, 0, nullptr, m->pa8, m->pab,
                                      pad8(m->pool_C), m->stats + pl * ST_PER_LAYER + 1, s));
        }
        if (m->speculate && L.pf_spec.rq_pred && !L.static_q) {
            // speculating: the contraction requantises with the predicted shift in its
            // epilogue; its re-launch checks the prediction against the max and returns at
            // once when it held, else recomputes with the step's shift (requantisation class,
            // no counted work)
            ITO_LAUNCH(m, s, ITO_PROF_GEMM, gemm_ops(L.pf_spec), gemm_run(L.pf_spec, s));
            ITO_LAUNCH(m, s, ITO_PROF_REQUANT, 0.0, gemm_run(L.pf_redo, s));
        } else {
            if (L.ig)
                ITO_LAUNCH(m, s, ITO_PROF_GEMM, 2.0 * L.rows_out * L.OC * L.K, conv_igemm_run(L.pig_f, s));
            else
                ITO_LAUNCH(m, s, ITO_PROF_GEMM, gemm_ops(L.pf), gemm_run(L.pf, s));
            if (L.static_q)
                ITO_LAUNCH(m, s, ITO_PROF_REQUANT, requant_bytes(L.rows_out * L.OC, L.ab != nullptr, false),
                           launch_requant_static(L.y32, L.rows_out, L.OC, L.off32, L.mult32, L.k32, L.relu ? 1 : 0,
                                                 L.a8, L.ab, L.lda, L.mask, s));
            else {
                // the logits' requantisation also writes the top error (the backward's first delta)
                const bool top = l == nl - 1 && labels;
                const TopErr te{labels, m->target_mag, L.e8, L.eb, L.lde, nullptr};
                ITO_LAUNCH(m, s, ITO_PROF_REQUANT,
                           requant_bytes(L.rows_out * L.OC, L.ab != nullptr, false) + (top ? 3.0 * B * L.OC : 0.0),
                           launch_requant(L.y32, L.rows_out, L.OC, m->umax(l, ST_YMAX), p.target_bits,
                                          L.relu ? 1 : 0, nullptr, L.a8, L.ab, L.lda, m->sval(l, ST_YS), s, nullptr,
                                          L.mask, m->last_y(l), top ? &te : nullptr));
                m->top_fused = top;
            }
        }
        in8 = L.a8;
    }
    return ITO_OK;
}

// Backward, top-down. Per layer: delta propagation with the pre-update weights (not
// for the first layer), its requantisation, the weight gradient, the update. With the
// overlap on, the contractions stay on `s` and the bandwidth passes go to the side
// stream `b`: requantising layer l's propagated delta runs beside layer l's weight
// gradient, and layer l's update beside layer l-1's delta propagation. Events order
// every read after its write: b waits for the delta-propagation result (delta ready)
// and for the weight gradient (before the update); s waits for the requantised delta
// before the next layer's contractions read it; s joins b at the end of the step.
// Backward in overlap mode 3: the delta chain (delta propagation, its requantisation, the
// next layer's delta propagation ...) on s; each layer's weight gradient and update on the
// second stream w, the weight gradient once its delta is ready (event ev_delta(l) on s), the
// update once the delta propagation that read the old weights is done (ev_dgrad(l)).
// The weight gradients use their own split-K workspace; the step ends joined on s.
static int model_backward_split(ito_model* m, cudaStream_t s)
{
    const int B = m->batch;
    const int nl = (int)m->L.size();
    const ito_niti_params p = m->p;
    cudaStream_t w = m->side;
    auto sync = [&](cudaEvent_t e, cudaStream_t from, cudaStream_t to) -> int {
        if (cudaEventRecord(e, from) != cudaSuccess || cudaStreamWaitEvent(to, e, 0) != cudaSuccess)
            return set_error(ITO_ERR_CUDA, "stream ordering event failed");
        return ITO_OK;
    };
    for (int l = nl - 1; l >= m->opt.trainable_from; --l) {
        MLayer& L = m->L[l];
        const bool conv = L.kind == ITO_LAYER_CONV3X3_RELU;
        ITO_TRY(sync(m->ev_delta(l), s, w));   // this layer's delta is ready
        if (L.ig)
            ITO_LAUNCH(m, w, ITO_PROF_GEMM, 2.0 * L.rows_out * L.OC * L.K, conv_igemm_run(L.pig_g, w));
        else
            ITO_LAUNCH(m, w, ITO_PROF_GEMM, gemm_ops(L.pg), gemm_run(L.pg, w));
        if (L.has_dgrad) {
            if (m->speculate && L.pd_spec.rq_pred) {
                ITO_LAUNCH(m, s, ITO_PROF_GEMM, gemm_ops(L.pd_spec), gemm_run(L.pd_spec, s));
                ITO_LAUNCH(m, s, ITO_PROF_REQUANT, 0.0, gemm_run(L.pd_redo, s));
            } else {
                if (L.s2)
                    ITO_LAUNCH(m, s, ITO_PROF_GEMM, 2.0 * L.rows_in * L.IC * 9 * L.OC / 4,
                               conv_dgrad_s2_run(L.ps2, s));
                else
                    ITO_LAUNCH(m, s, ITO_PROF_GEMM, gemm_ops(L.pd), gemm_run(L.pd, s));
            }
            // the update below may overwrite the weights once this delta propagation is done
            ITO_TRY(sync(m->ev_dgrad(l), s, w));
            if (!(m->speculate && L.pd_spec.rq_pred)) {
                MLayer& prev = m->L[l - 1];
                if (conv) {
                    if (!L.s2)
                        ITO_LAUNCH(m, s, ITO_PROF_OTHER, 4.0 * L.rows_out * L.K + 4.0 * L.rows_in * L.IC,
                                   launch_col2im(L.dcol, B, L.H, L.W, L.IC, L.OH, L.OW, L.stride, L.d32,
                                                 m->umax(l, ST_DMAX), s));
                    ITO_LAUNCH(m, s, ITO_PROF_REQUANT, requant_bytes(L.rows_in * L.IC, true, true),
                               launch_requant(L.d32, L.rows_in, L.IC, m->umax(l, ST_DMAX), p.target_bits, 0,
                                              prev.mask ? nullptr : prev.a8, prev.e8, prev.eb, prev.lde,
                                              m->sval(l, ST_DS), s, prev.mask, nullptr));
                } else if (l == m->n_conv && m->has_pool) {
                    ITO_LAUNCH(m, s, ITO_PROF_REQUANT, requant_bytes((int64_t)B * L.IC, false, false),
                               launch_requant(L.d32, B, L.IC, m->umax(l, ST_DMAX), p.target_bits, 0, nullptr, m->pe8,
                                              nullptr, 0, m->sval(l, ST_DS), s));
                    ITO_LAUNCH(m, s, ITO_PROF_OTHER, 4.0 * B * m->pool_HW * m->pool_C,
                               launch_gap_bwd(m->pe8, prev.a8, B, m->pool_HW, m->pool_C, prev.e8, prev.eb, s));
                } else {
                    ITO_LAUNCH(m, s, ITO_PROF_REQUANT, requant_bytes((int64_t)B * L.IC, true, prev.relu),
                               launch_requant(L.d32, B, L.IC, m->umax(l, ST_DMAX), p.target_bits, 0,
                                              (prev.relu && !prev.mask) ? prev.a8 : nullptr, prev.e8, prev.eb,
                                              prev.lde, m->sval(l, ST_DS), s, prev.mask, nullptr, m->last_d(l)));
                }
            }
        }
        // G read (4 B), W read and written (1 + 1 B), bf16 copy written (2 B)
        ITO_LAUNCH(m, w, ITO_PROF_UPDATE, 8.0 * L.OC * L.K,
                   launch_niti_update(L.W8, L.Wb, L.ldw, L.g32, L.OC, L.K, m->umax(l, ST_GMAX), p.target_bits,
                                      p.mu_weight, m->sval(l, ST_GS), m->sval(l, ST_WS),
                                      reinterpret_cast<uint32_t*>(m->sval(l, ST_NZ)), w));
    }
    return sync(m->ev_join(), w, s);
}

static int model_backward(ito_model* m, const int8_t* x, const int32_t* labels, cudaStream_t s)
{
    const int B = m->batch;
    const int nl = (int)m->L.size();
    const ito_niti_params p = m->p;
    // b: the update stream; r_side: the stream of the delta requantisation
    cudaStream_t b = m->overlap ? m->side : s;
    cudaStream_t r_side = m->overlap == 1 ? m->side : s;
    auto sync = [&](cudaEvent_t e, cudaStream_t from, cudaStream_t to) -> int {
        if (from == to) return ITO_OK;
        if (cudaEventRecord(e, from) != cudaSuccess || cudaStreamWaitEvent(to, e, 0) != cudaSuccess)
            return set_error(ITO_ERR_CUDA, "stream ordering event failed");
        return ITO_OK;
    };
    MLayer& top = m->L[nl - 1];
    if (!m->top_fused)
        ITO_LAUNCH(m, s, ITO_PROF_OTHER, 4.0 * B * top.OC + 4.0 * B,
                   launch_top_error(top.a8, labels, B, top.OC, m->target_mag, top.e8, top.eb, top.lde, s));
    ITO_TRY(sync(m->ev_fork(), s, b));
    if (m->overlap == 3) return model_backward_split(m, s);
    bool delta_on_side = false;   // the layer above requantised this layer's delta on the side stream
    for (int l = nl - 1; l >= m->opt.trainable_from; --l) {
        MLayer& L = m->L[l];
        const bool conv = L.kind == ITO_LAYER_CONV3X3_RELU;
        // this layer's delta (produced on the side stream by the layer above) before its contractions
        if (delta_on_side && cudaStreamWaitEvent(s, m->ev_delta(l + 1), 0) != cudaSuccess)
            return set_error(ITO_ERR_CUDA, "stream ordering event failed");
        delta_on_side = false;
        if (L.has_dgrad && m->speculate && L.pd_spec.rq_pred) {
            // speculating delta propagation and its re-launch, both on s (as in the forward)
            ITO_LAUNCH(m, s, ITO_PROF_GEMM, gemm_ops(L.pd_spec), gemm_run(L.pd_spec, s));
            ITO_LAUNCH(m, s, ITO_PROF_REQUANT, 0.0, gemm_run(L.pd_redo, s));
        } else if (L.has_dgrad) {
            if (L.s2)
                ITO_LAUNCH(m, s, ITO_PROF_GEMM, 2.0 * L.rows_in * L.IC * 9 * L.OC / 4,
                           conv_dgrad_s2_run(L.ps2, s));
            else
                ITO_LAUNCH(m, s, ITO_PROF_GEMM, gemm_ops(L.pd), gemm_run(L.pd, s));
            const cudaStream_t r = r_side;
            ITO_TRY(sync(m->ev_dgrad(l), s, r));   // the propagated delta is complete
            MLayer& prev = m->L[l - 1];
            if (conv) {
                if (!L.s2)
                    ITO_LAUNCH(m, r, ITO_PROF_OTHER, 4.0 * L.rows_out * L.K + 4.0 * L.rows_in * L.IC,
                               launch_col2im(L.dcol, B, L.H, L.W, L.IC, L.OH, L.OW, L.stride, L.d32,
                                             m->umax(l, ST_DMAX), r));
                ITO_LAUNCH(m, r, ITO_PROF_REQUANT, requant_bytes(L.rows_in * L.IC, true, true),
                           launch_requant(L.d32, L.rows_in, L.IC, m->umax(l, ST_DMAX), p.target_bits, 0,
                                          prev.mask ? nullptr : prev.a8, prev.e8, prev.eb, prev.lde,
                                          m->sval(l, ST_DS), r, prev.mask, nullptr));
            } else if (l == m->n_conv && m->has_pool) {
                // pooled delta (the pooled activation has no ReLU), then the pooling backward
                ITO_LAUNCH(m, r, ITO_PROF_REQUANT, requant_bytes((int64_t)B * L.IC, false, false),
                           launch_requant(L.d32, B, L.IC, m->umax(l, ST_DMAX), p.target_bits, 0, nullptr, m->pe8,
                                          nullptr, 0, m->sval(l, ST_DS), r));
                ITO_LAUNCH(m, r, ITO_PROF_OTHER, 4.0 * B * m->pool_HW * m->pool_C,
                           launch_gap_bwd(m->pe8, prev.a8, B, m->pool_HW, m->pool_C, prev.e8, prev.eb, r));
            } else {
                ITO_LAUNCH(m, r, ITO_PROF_REQUANT, requant_bytes((int64_t)B * L.IC, true, prev.relu),
                           launch_requant(L.d32, B, L.IC, m->umax(l, ST_DMAX), p.target_bits, 0,
                                          (prev.relu && !prev.mask) ? prev.a8 : nullptr, prev.e8, prev.eb, prev.lde,
                                          m->sval(l, ST_DS), r, prev.mask, nullptr, m->last_d(l)));
            }
            if (r != s) {
                if (cudaEventRecord(m->ev_delta(l), r) != cudaSuccess)
                    return set_error(ITO_ERR_CUDA, "stream ordering event failed");
                delta_on_side = true;
            }
        }
        if (L.ig)
            ITO_LAUNCH(m, s, ITO_PROF_GEMM, 2.0 * L.rows_out * L.OC * L.K, conv_igemm_run(L.pig_g, s));
        else
            ITO_LAUNCH(m, s, ITO_PROF_GEMM, gemm_ops(L.pg), gemm_run(L.pg, s));
        ITO_TRY(sync(m->ev_wgrad(l), s, b));       // the weight gradient is complete
        // G read (4 B), W read and written (1 + 1 B), bf16 copy written (2 B)
        ITO_LAUNCH(m, b, ITO_PROF_UPDATE, 8.0 * L.OC * L.K,
                   launch_niti_update(L.W8, L.Wb, L.ldw, L.g32, L.OC, L.K, m->umax(l, ST_GMAX), p.target_bits,
                                      p.mu_weight, m->sval(l, ST_GS), m->sval(l, ST_WS),
                                      reinterpret_cast<uint32_t*>(m->sval(l, ST_NZ)), b));
        // the offsets' gradient reads this layer's delta, whose (ping-pong) buffer the next
        // requantisation overwrites: it runs on the requantisation stream, before that one
        if (L.static_q)
            ITO_LAUNCH(m, r_side, ITO_PROF_UPDATE, (double)L.rows_out * L.OC + 12.0 * L.OC,
                       launch_offset_grad_update(L.e8, L.rows_out, L.OC, L.og32, m->umax(l, ST_OGMAX), L.off32,
                                                 p.target_bits, p.mu_weight, m->sval(l, ST_OGS), m->sval(l, ST_OWS),
                                                 reinterpret_cast<uint32_t*>(m->sval(l, ST_ONZ)), r_side));
    }
    ITO_TRY(sync(m->ev_join(), b, s));
    (void)x;
    return ITO_OK;
}

extern "C" {

int ito_model_create(const ito_layer_desc* layers, int n_layers, int batch, ito_niti_params p, int32_t target_mag,
                     ito_model** out)
{
    return ito_model_create_ex(layers, n_layers, batch, p, target_mag, nullptr, out);
}

int ito_model_create_ex(const ito_layer_desc* layers, int n_layers, int batch, ito_niti_params p,
                        int32_t target_mag, const ito_model_options* opt, ito_model** out)
{
    if (!layers || !out || n_layers < 1) return set_error(ITO_ERR_ARG, "NULL layers/out or no layers");
    if (batch < 1 || batch > (1 << 20)) return set_error(ITO_ERR_SHAPE, "batch");
    if (p.target_bits < 1 || p.target_bits > 8 || p.mu_weight < 0 || p.mu_weight > 31)
        return set_error(ITO_ERR_ARG, "NITI parameters out of range");
    *out = nullptr;
    ito_model* m = new ito_model();
    m->batch = batch;
    m->p = p;
    m->target_mag = target_mag;
    if (opt) m->opt = *opt;
    int r = build_model(m, layers, n_layers);
    if (r != ITO_OK) {
        ito_model_destroy(m);
        return r;
    }
    *out = m;
    return ITO_OK;
}

static void drop_graphs(ito_model* m)
{
    for (auto& g : m->graphs) cudaGraphExecDestroy(g.exec);
    m->graphs.clear();
    m->graph_warm = false;
}

int ito_model_destroy(ito_model* m)
{
    if (!m) return ITO_OK;
    cudaDeviceSynchronize();
    drop_graphs(m);
    for (cudaEvent_t e : m->prof_ev) cudaEventDestroy(e);
    for (cudaEvent_t e : m->sync_ev) cudaEventDestroy(e);
    for (int i = 0; i < 2; ++i) {
        if (m->ev_copied[i]) cudaEventDestroy(m->ev_copied[i]);
        if (m->ev_consumed[i]) cudaEventDestroy(m->ev_consumed[i]);
    }
    if (m->side) cudaStreamDestroy(m->side);
    if (m->copy_stream) cudaStreamDestroy(m->copy_stream);
    for (void* p : m->allocs) cudaFree(p);
    delete m;
    return ITO_OK;
}

static int weight_layer(const ito_model* m, int layer)
{
    if (!m || layer < 0 || layer >= (int)m->L.size()) return -1;
    return layer;
}

int ito_model_set_weights(ito_model* m, int layer, const int8_t* W, int on_host, void* stream)
{
    const int l = weight_layer(m, layer);
    if (l < 0 || !W) return set_error(ITO_ERR_ARG, "bad model, layer or W");
    MLayer& L = m->L[l];
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t bytes = (size_t)L.OC * L.K;
    cudaError_t e = cudaMemcpyAsync(L.W8, W, bytes, on_host ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return set_error(ITO_ERR_CUDA, "weight copy: %s", cudaGetErrorString(e));
    ITO_TRY(launch_i8_to_bf16(L.W8, L.OC, L.K, L.Wb, L.ldw, s));
    if (on_host && cudaStreamSynchronize(s) != cudaSuccess) return set_error(ITO_ERR_CUDA, "sync");
    return ITO_OK;
}

int ito_model_get_weights(const ito_model* m, int layer, int8_t* W, int on_host, void* stream)
{
    const int l = weight_layer(m, layer);
    if (l < 0 || !W) return set_error(ITO_ERR_ARG, "bad model, layer or W");
    const MLayer& L = m->L[l];
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(W, L.W8, (size_t)L.OC * L.K,
                                    on_host ? cudaMemcpyDeviceToHost : cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return set_error(ITO_ERR_CUDA, "weight copy: %s", cudaGetErrorString(e));
    if (on_host && cudaStreamSynchronize(s) != cudaSuccess) return set_error(ITO_ERR_CUDA, "sync");
    return ITO_OK;
}

int ito_model_tensor(const ito_model* m, const char* name, void** dev_ptr, int* elem_bytes, int64_t* numel)
{
    if (!m || !name || !dev_ptr || !elem_bytes || !numel) return set_error(ITO_ERR_ARG, "NULL argument");
    const int nl = (int)m->L.size();
    auto put = [&](const void* p, int eb, int64_t n) {
        *dev_ptr = const_cast<void*>(p);
        *elem_bytes = eb;
        *numel = n;
        return p ? ITO_OK : set_error(ITO_ERR_ARG, "tensor %s does not exist in this model", name);
    };
    const std::string s(name);
    if (s == "stats") return put(m->stats, 4, m->n_stats);
    if (s == "x") return put(m->x8, 1, (int64_t)m->batch * m->in_features);
    if (s == "labels") return put(m->labels, 4, m->batch);
    if (s == "p") return put(m->p32, 4, (int64_t)m->batch * m->pool_C);
    if (s == "pa") return put(m->pa8, 1, (int64_t)m->batch * m->pool_C);
    if (s == "pe") return put(m->pe8, 1, (int64_t)m->batch * m->pool_C);
    if (s == "spec") return put(m->spec, 4, 8 * (int64_t)nl);
    if (s == "spec_count") return put(m->spec_count, 8, 2);
    // per-layer tensors: a name prefix followed by the layer index
    size_t pos = 0;
    while (pos < s.size() && (s[pos] < '0' || s[pos] > '9')) ++pos;
    if (pos == 0 || pos == s.size()) return set_error(ITO_ERR_ARG, "unknown tensor name %s", name);
    char* end = nullptr;
    const long l = strtol(s.c_str() + pos, &end, 10);
    if (!end || *end || l < 0 || l >= nl) return set_error(ITO_ERR_ARG, "unknown tensor name %s", name);
    const MLayer& L = m->L[l];
    const std::string key = s.substr(0, pos);
    if (key == "y") return put(L.y32, 4, L.rows_out * L.OC);
    if (key == "a") return put(L.a8, 1, L.rows_out * L.OC);
    if (key == "e") return put(L.e8, 1, L.rows_out * L.OC);
    if (key == "d") return put(L.d32, 4, L.rows_in * L.IC);
    if (key == "g") return put(L.g32, 4, (int64_t)L.OC * L.K);
    if (key == "w") return put(L.W8, 1, (int64_t)L.OC * L.K);
    if (key == "m") return put(L.mask, 1, L.rows_out * (L.OC / 8));
    if (key == "off") return put(L.off32, 4, L.OC);
    if (key == "og") return put(L.og32, 4, L.OC);
    return set_error(ITO_ERR_ARG, "unknown tensor name %s", name);
}

int ito_model_set_static_requant(ito_model* m, int layer, const int32_t* offset, const int32_t* mult,
                                 const int32_t* shift, int on_host, void* stream)
{
    const int l = weight_layer(m, layer);
    if (l < 0 || !offset || !mult || !shift) return set_error(ITO_ERR_ARG, "bad model, layer or array");
    MLayer& L = m->L[l];
    if (!L.off32) return set_error(ITO_ERR_UNSUPPORTED, "static requantisation is for Linear layers");
    if (on_host) {
        for (int c = 0; c < L.OC; ++c)
            if (shift[c] < 0 || shift[c] > 62) return set_error(ITO_ERR_ARG, "shift[%d] outside 0..62", c);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const cudaMemcpyKind kind = on_host ? cudaMemcpyHostToDevice : cudaMemcpyDeviceToDevice;
    const size_t bytes = sizeof(int32_t) * L.OC;
    if (cudaMemcpyAsync(L.off32, offset, bytes, kind, s) != cudaSuccess ||
        cudaMemcpyAsync(L.mult32, mult, bytes, kind, s) != cudaSuccess ||
        cudaMemcpyAsync(L.k32, shift, bytes, kind, s) != cudaSuccess)
        return set_error(ITO_ERR_CUDA, "static requant copy failed");
    if (on_host && cudaStreamSynchronize(s) != cudaSuccess) return set_error(ITO_ERR_CUDA, "sync");
    L.static_q = true;
    if (L.pf_spec.rq_pred) {
        // the static requantisation replaces the dynamic shift: the forward slot no longer speculates
        const int32_t zero = 0;
        if (cudaDeviceSynchronize() != cudaSuccess ||
            cudaMemcpy(m->spec + 4 * (int)m->L.size() + l, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
            return set_error(ITO_ERR_CUDA, "speculation flag update failed");
        L.pf_spec = L.pf;
        L.pf_redo = GemmPlan{};
    }
    drop_graphs(m);
    return ITO_OK;
}

int ito_model_stat_index(const ito_model* m, const char* name)
{
    if (!m || !name) return -1;
    for (auto& kv : m->stat_names)
        if (kv.first == name) return kv.second;
    return -1;
}

int ito_model_num_stats(const ito_model* m) { return m ? m->n_stats : 0; }

int ito_model_profile(ito_model* m, int enable)
{
    if (!m) return set_error(ITO_ERR_ARG, "NULL model");
    if (cudaDeviceSynchronize() != cudaSuccess) return set_error(ITO_ERR_CUDA, "sync");
    // graphs captured with and without timing events differ
    drop_graphs(m);
    m->prof_on = enable != 0;
    m->prof_n = 0;
    m->prof_cls.clear();
    m->prof_work.clear();
    if (m->prof_on) m->grow_events(256);
    return ITO_OK;
}

int ito_model_profile_read(ito_model* m, double* ms, double* work, int64_t* launches)
{
    if (!m || !ms || !work || !launches) return set_error(ITO_ERR_ARG, "NULL argument");
    for (int c = 0; c < ITO_PROF_NCLASS; ++c) {
        ms[c] = 0;
        work[c] = 0;
        launches[c] = 0;
    }
    for (int i = 0; i < m->prof_n; ++i) {
        float t = 0;
        if (cudaEventSynchronize(m->prof_ev[2 * i + 1]) != cudaSuccess ||
            cudaEventElapsedTime(&t, m->prof_ev[2 * i], m->prof_ev[2 * i + 1]) != cudaSuccess)
            return set_error(ITO_ERR_CUDA, "profile event read failed");
        ms[m->prof_cls[i]] += t;
        work[m->prof_cls[i]] += m->prof_work[i];
        launches[m->prof_cls[i]] += 1;
    }
    m->prof_n = 0;
    m->prof_cls.clear();
    m->prof_work.clear();
    return ITO_OK;
}

int ito_model_kernels_per_step(const ito_model* m) { return m ? m->launches : 0; }

int ito_model_set_speculation(ito_model* m, int enable)
{
    if (!m) return set_error(ITO_ERR_ARG, "NULL model");
    if ((enable != 0) != m->speculate) {
        if (cudaDeviceSynchronize() != cudaSuccess) return set_error(ITO_ERR_CUDA, "sync");
        drop_graphs(m);   // captured steps encode the setting
        m->speculate = enable != 0;
    }
    return ITO_OK;
}

int ito_model_get_speculation(const ito_model* m, int* enabled)
{
    if (!m || !enabled) return set_error(ITO_ERR_ARG, "NULL argument");
    *enabled = m->speculate ? 1 : 0;
    return ITO_OK;
}

int ito_model_get_overlap(const ito_model* m, int* mode)
{
    if (!m || !mode) return set_error(ITO_ERR_ARG, "NULL argument");
    *mode = m->overlap;
    return ITO_OK;
}

int ito_model_set_overlap(ito_model* m, int mode)
{
    if (!m || mode < 0 || mode > 3) return set_error(ITO_ERR_ARG, "bad model or overlap mode");
    if (mode == 3 && !m->overlap3_ok)
        return set_error(ITO_ERR_UNSUPPORTED, "overlap mode 3 needs unshared delta buffers and dynamic requantisation");
    if (mode != m->overlap) {
        if (cudaDeviceSynchronize() != cudaSuccess) return set_error(ITO_ERR_CUDA, "sync");
        drop_graphs(m);   // captured steps encode the stream layout
        m->overlap = mode;
    }
    return ITO_OK;
}

int ito_model_use_graphs(ito_model* m, int enable)
{
    if (!m) return set_error(ITO_ERR_ARG, "NULL model");
    if (cudaDeviceSynchronize() != cudaSuccess) return set_error(ITO_ERR_CUDA, "sync");
    drop_graphs(m);
    m->graph_on = enable != 0;
    return ITO_OK;
}

static int step_direct(ito_model* m, const int8_t* x, const int32_t* labels, cudaStream_t s)
{
    m->launches = 0;
    // statistics zeroed, this step's shift predictions = the last step's shifts, input in bf16
    ITO_TRY(model_begin(m, x, true, s));
    ITO_TRY(model_forward(m, x, labels, s));
    return model_backward(m, x, labels, s);
}

int ito_train_step(ito_model* m, const int8_t* x, const int32_t* labels, void* stream)
{
    if (!m || !x || !labels) return set_error(ITO_ERR_ARG, "NULL argument");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // graphs need a capturable (non-default) stream
    if (!m->graph_on || s == nullptr) return step_direct(m, x, labels, s);
    for (auto& g : m->graphs)
        if (g.x == x && g.labels == labels) {
            m->launches = g.launches;
            if (m->prof_on) {
                // the replay re-records the graph's timing events: the last replay's timings are readable
                m->prof_n = (int)g.prof_cls.size();
                m->prof_cls = g.prof_cls;
                m->prof_work = g.prof_work;
            }
            cudaError_t e = cudaGraphLaunch(g.exec, s);
            return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "graph launch: %s", cudaGetErrorString(e));
        }
    if (!m->graph_warm) {
        // one direct step first: kernel attributes and tensor maps are set up outside any capture
        m->graph_warm = true;
        return step_direct(m, x, labels, s);
    }
    if (m->graphs.size() >= 8) {
        drop_graphs(m);
        m->graph_warm = true;
    }
    // timing events of earlier direct steps are read before capture reuses the pool
    if (m->prof_on && m->prof_n > 0 && cudaStreamSynchronize(s) != cudaSuccess)
        return set_error(ITO_ERR_CUDA, "sync before capture");
    m->prof_n = 0;
    m->prof_cls.clear();
    m->prof_work.clear();
    cudaError_t e = cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return set_error(ITO_ERR_CUDA, "begin capture: %s", cudaGetErrorString(e));
    m->capturing = true;
    const int r = step_direct(m, x, labels, s);
    m->capturing = false;
    cudaGraph_t graph = nullptr;
    e = cudaStreamEndCapture(s, &graph);
    if (r != ITO_OK) {
        if (graph) cudaGraphDestroy(graph);
        return r;
    }
    if (e != cudaSuccess) return set_error(ITO_ERR_CUDA, "end capture: %s", cudaGetErrorString(e));
    cudaGraphExec_t exec = nullptr;
    e = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return set_error(ITO_ERR_CUDA, "graph instantiate: %s", cudaGetErrorString(e));
    m->graphs.push_back({x, labels, exec, m->launches, m->prof_cls, m->prof_work});
    e = cudaGraphLaunch(exec, s);
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "graph launch: %s", cudaGetErrorString(e));
}

int ito_train_step_host(ito_model* m, const int8_t* x_host, const int32_t* labels_host, int32_t* stats_host,
                        void* stream)
{
    if (!m || !x_host || !labels_host) return set_error(ITO_ERR_ARG, "NULL argument");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(m->x8, x_host, (size_t)m->batch * m->in_features, cudaMemcpyHostToDevice, s);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(m->labels, labels_host, sizeof(int32_t) * m->batch, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return set_error(ITO_ERR_CUDA, "input copy: %s", cudaGetErrorString(e));
    ITO_TRY(ito_train_step(m, m->x8, m->labels, stream));
    if (stats_host) {
        e = cudaMemcpyAsync(stats_host, m->stats, sizeof(int32_t) * m->n_stats, cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) return set_error(ITO_ERR_CUDA, "stats copy: %s", cudaGetErrorString(e));
    }
    e = cudaStreamSynchronize(s);
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "step: %s", cudaGetErrorString(e));
}

int ito_train_step_host_async(ito_model* m, const int8_t* x_host, const int32_t* labels_host, int32_t* stats_host,
                              void* stream)
{
    if (!m || !x_host || !labels_host) return set_error(ITO_ERR_ARG, "NULL argument");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int i = (int)(m->async_steps & 1);
    int8_t* xd = i ? m->x8b : m->x8;
    int32_t* ld = i ? m->labels_b : m->labels;
    // the copy waits for the step that last read this buffer, and the step for the copy
    cudaError_t e = cudaStreamWaitEvent(m->copy_stream, m->ev_consumed[i], 0);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(xd, x_host, (size_t)m->batch * m->in_features, cudaMemcpyHostToDevice, m->copy_stream);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(ld, labels_host, sizeof(int32_t) * m->batch, cudaMemcpyHostToDevice, m->copy_stream);
    if (e == cudaSuccess) e = cudaEventRecord(m->ev_copied[i], m->copy_stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, m->ev_copied[i], 0);
    if (e != cudaSuccess) return set_error(ITO_ERR_CUDA, "input copy: %s", cudaGetErrorString(e));
    ITO_TRY(ito_train_step(m, xd, ld, stream));
    if (stats_host) {
        e = cudaMemcpyAsync(stats_host, m->stats, sizeof(int32_t) * m->n_stats, cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) return set_error(ITO_ERR_CUDA, "stats copy: %s", cudaGetErrorString(e));
    }
    e = cudaEventRecord(m->ev_consumed[i], s);
    if (e != cudaSuccess) return set_error(ITO_ERR_CUDA, "event: %s", cudaGetErrorString(e));
    ++m->async_steps;
    return ITO_OK;
}

int ito_infer(ito_model* m, const int8_t* x, int8_t* logits, void* stream)
{
    if (!m || !x || !logits) return set_error(ITO_ERR_ARG, "NULL argument");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    m->launches = 0;
    ITO_TRY(model_begin(m, x, false, s));
    ITO_TRY(model_forward(m, x, nullptr, s));
    const MLayer& top = m->L.back();
    cudaError_t e = cudaMemcpyAsync(logits, top.a8, (size_t)top.rows_out * top.OC, cudaMemcpyDeviceToDevice, s);
    return e == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "logits copy: %s", cudaGetErrorString(e));
}

static const uint32_t kMagic = 0x3249544fu;   // "OTI2": weights, then per Linear layer a static flag and offsets

int ito_model_save(const ito_model* m, const char* path)
{
    if (!m || !path) return set_error(ITO_ERR_ARG, "NULL argument");
    if (cudaDeviceSynchronize() != cudaSuccess) return set_error(ITO_ERR_CUDA, "sync");
    FILE* f = fopen(path, "wb");
    if (!f) return set_error(ITO_ERR_ARG, "cannot open %s", path);
    const uint32_t n = (uint32_t)m->L.size();
    bool ok = fwrite(&kMagic, 4, 1, f) == 1 && fwrite(&n, 4, 1, f) == 1;
    std::vector<int8_t> buf;
    for (const MLayer& L : m->L) {
        const int64_t shape[2] = {L.OC, L.K};
        ok = ok && fwrite(shape, 8, 2, f) == 2;
    }
    for (const MLayer& L : m->L) {
        buf.resize((size_t)L.OC * L.K);
        ok = ok && cudaMemcpy(buf.data(), L.W8, buf.size(), cudaMemcpyDeviceToHost) == cudaSuccess;
        ok = ok && fwrite(buf.data(), 1, buf.size(), f) == buf.size();
    }
    std::vector<int32_t> o;
    for (const MLayer& L : m->L) {
        const int32_t flag = L.static_q ? 1 : 0;
        ok = ok && fwrite(&flag, 4, 1, f) == 1;
        if (!flag) continue;
        for (const int32_t* src : {L.off32, L.mult32, L.k32}) {
            o.resize(L.OC);
            ok = ok && cudaMemcpy(o.data(), src, 4 * o.size(), cudaMemcpyDeviceToHost) == cudaSuccess;
            ok = ok && fwrite(o.data(), 4, o.size(), f) == o.size();
        }
    }
    fclose(f);
    return ok ? ITO_OK : set_error(ITO_ERR_ARG, "write to %s failed", path);
}

int ito_model_load(ito_model* m, const char* path)
{
    if (!m || !path) return set_error(ITO_ERR_ARG, "NULL argument");
    FILE* f = fopen(path, "rb");
    if (!f) return set_error(ITO_ERR_ARG, "cannot open %s", path);
    uint32_t magic = 0, n = 0;
    bool ok = fread(&magic, 4, 1, f) == 1 && fread(&n, 4, 1, f) == 1 && magic == kMagic && n == m->L.size();
    for (const MLayer& L : m->L) {
        int64_t shape[2] = {0, 0};
        ok = ok && fread(shape, 8, 2, f) == 2 && shape[0] == L.OC && shape[1] == L.K;
    }
    std::vector<int8_t> buf;
    for (size_t l = 0; ok && l < m->L.size(); ++l) {
        MLayer& L = m->L[l];
        buf.resize((size_t)L.OC * L.K);
        ok = fread(buf.data(), 1, buf.size(), f) == buf.size();
        ok = ok && ito_model_set_weights(m, (int)l, buf.data(), 1, nullptr) == ITO_OK;
    }
    for (size_t l = 0; ok && l < m->L.size(); ++l) {
        MLayer& L = m->L[l];
        int32_t flag = 0;
        ok = fread(&flag, 4, 1, f) == 1;
        if (!ok || !flag) continue;
        std::vector<int32_t> off(L.OC), mult(L.OC), k(L.OC);
        ok = fread(off.data(), 4, L.OC, f) == (size_t)L.OC && fread(mult.data(), 4, L.OC, f) == (size_t)L.OC &&
             fread(k.data(), 4, L.OC, f) == (size_t)L.OC;
        ok = ok && ito_model_set_static_requant(m, (int)l, off.data(), mult.data(), k.data(), 1, nullptr) == ITO_OK;
    }
    fclose(f);
    if (!ok) return set_error(ITO_ERR_SHAPE, "checkpoint %s does not match the model", path);
    return cudaDeviceSynchronize() == cudaSuccess ? ITO_OK : set_error(ITO_ERR_CUDA, "sync");
}

}  // extern "C"
