// graph.cu — bucketed CUDA-graph executor for small-batch decode steps.
//
// "mini-llm-inference-engine" README, architecture overview (core design principles:
// CUDA Graph multi-bucket capture).  A decode step at small batch is a handful of
// microsecond-scale kernels whose launches cost as much as their work.  The executor
// records the step (per layer: append + decode, or the fused decode step) once for each
// batch-size bucket through the public entry points, on an internal stream under
// thread-local stream capture, and replays the smallest bucket that holds a launch's
// sequences with a single cudaGraphLaunch.  Buffers are captured by address; padding rows
// of a bucket are kept inert by the caller (length 0, slot -1).
#include <cuda_runtime.h>

#include <new>

#include "internal.h"
#include "nvtx.h"
#include "pkv.h"

struct pkv_decode_graph {
  int device = 0;
  int num_buckets = 0;
  int buckets[PKV_GRAPH_MAX_BUCKETS] = {};
  cudaGraphExec_t exec[PKV_GRAPH_MAX_BUCKETS] = {};
};

namespace {

pkv_status check_desc(const pkv_decode_graph_desc* d) {
  if (!d || !d->layers || !d->buckets) return PKV_ERR_NULL;
  if (d->num_layers < 1 || d->num_buckets < 1 || d->num_buckets > PKV_GRAPH_MAX_BUCKETS)
    return PKV_ERR_SHAPE;
  for (int i = 0; i < d->num_buckets; ++i)
    if (d->buckets[i] < 1 || (i > 0 && d->buckets[i] <= d->buckets[i - 1])) return PKV_ERR_SHAPE;
  bool appends = false;
  for (int l = 0; l < d->num_layers; ++l) appends |= d->layers[l].k_new != nullptr;
  if ((appends || d->fused) && !d->slot_mapping) return PKV_ERR_NULL;
  return PKV_OK;
}

// The calls of one step for the first B sequences, on stream st.
pkv_status record_step(const pkv_decode_graph_desc* d, int B, cudaStream_t st) {
  for (int l = 0; l < d->num_layers; ++l) {
    const pkv_graph_layer& L = d->layers[l];
    pkv_status s;
    if (d->fused) {
      s = pkv_decode_step(&L.cache, L.q, d->q_dtype, L.k_new, L.v_new, d->new_dtype,
                          d->slot_mapping, d->positions, d->rope_theta, B, d->num_q_heads,
                          d->block_tables, d->max_blocks_per_seq, d->context_lens, d->scale,
                          L.out, d->workspace, d->workspace_bytes, d->dev_status, st);
    } else {
      s = PKV_OK;
      if (L.k_new)
        s = pkv_append(&L.cache, L.k_new, L.v_new, d->new_dtype, d->slot_mapping, B,
                       d->dev_status, st);
      if (s == PKV_OK)
        s = pkv_decode_attn(&L.cache, L.q, d->q_dtype, B, d->num_q_heads, d->block_tables,
                            d->max_blocks_per_seq, d->context_lens, d->scale, L.out,
                            d->workspace, d->workspace_bytes, d->dev_status, st);
    }
    if (s != PKV_OK) return s;
  }
  return PKV_OK;
}

}  // namespace

extern "C" {

pkv_status pkv_decode_graph_workspace_size(const pkv_decode_graph_desc* d, size_t* bytes) {
  if (!bytes) return PKV_ERR_NULL;
  *bytes = 0;
  pkv_status s = check_desc(d);
  if (s != PKV_OK) return s;
  size_t need = 0;
  for (int l = 0; l < d->num_layers; ++l)
    for (int i = 0; i < d->num_buckets; ++i) {
      size_t n = 0;
      s = pkv_decode_workspace_size(&d->layers[l].cache, d->buckets[i], d->num_q_heads,
                                    d->max_blocks_per_seq, &n);
      if (s != PKV_OK) return s;
      if (n > need) need = n;
    }
  *bytes = need;
  return PKV_OK;
}

pkv_status pkv_decode_graph_create(const pkv_decode_graph_desc* d, pkv_decode_graph** out) {
  if (!out) return PKV_ERR_NULL;
  *out = nullptr;
  size_t need = 0;
  // validates the descriptor and every layer's cache, and plans every bucket (device
  // facts are queried here, outside the capture)
  pkv_status s = pkv_decode_graph_workspace_size(d, &need);
  if (s != PKV_OK) return s;
  if (need > 0 && (!d->workspace || d->workspace_bytes < need)) return PKV_ERR_WORKSPACE;
  pkv_decode_graph* g = new (std::nothrow) pkv_decode_graph();
  if (!g) return PKV_ERR_LAUNCH;
  if (cudaGetDevice(&g->device) != cudaSuccess) {
    delete g;
    return PKV_ERR_DEVICE;
  }
  cudaStream_t cs = nullptr;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) {
    delete g;
    return PKV_ERR_LAUNCH;
  }
  for (int i = 0; i < d->num_buckets && s == PKV_OK; ++i) {
    cudaGraph_t graph = nullptr;
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
      s = PKV_ERR_LAUNCH;
      break;
    }
    s = record_step(d, d->buckets[i], cs);
    // the capture always ends, whatever the recorded calls returned
    const cudaError_t e = cudaStreamEndCapture(cs, &graph);
    if (s == PKV_OK && (e != cudaSuccess || !graph)) s = PKV_ERR_LAUNCH;
    if (s == PKV_OK && cudaGraphInstantiate(&g->exec[i], graph, 0) != cudaSuccess) {
      g->exec[i] = nullptr;
      s = PKV_ERR_LAUNCH;
    }
    if (graph) cudaGraphDestroy(graph);
    if (s == PKV_OK) {
      g->buckets[i] = d->buckets[i];
      g->num_buckets = i + 1;
    }
  }
  cudaStreamDestroy(cs);
  if (s != PKV_OK) {
    pkv_decode_graph_destroy(g);
    (void)cudaGetLastError();  // a failed capture leaves no sticky error behind
    return s;
  }
  *out = g;
  return PKV_OK;
}

int32_t pkv_decode_graph_bucket(const pkv_decode_graph* g, int32_t num_seqs) {
  if (!g || num_seqs < 1) return 0;
  for (int i = 0; i < g->num_buckets; ++i)
    if (g->buckets[i] >= num_seqs) return g->buckets[i];
  return 0;
}

pkv_status pkv_decode_graph_launch(pkv_decode_graph* g, int32_t num_seqs, void* stream) {
  PKV_RANGE("pkv_decode_graph_launch");
  if (!g) return PKV_ERR_NULL;
  if (num_seqs < 0) return PKV_ERR_SHAPE;
  if (num_seqs == 0) return PKV_OK;
  int i = 0;
  while (i < g->num_buckets && g->buckets[i] < num_seqs) ++i;
  if (i == g->num_buckets) return PKV_ERR_SHAPE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != g->device) return PKV_ERR_DEVICE;
  return cudaGraphLaunch(g->exec[i], static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PKV_OK
             : PKV_ERR_LAUNCH;
}

void pkv_decode_graph_destroy(pkv_decode_graph* g) {
  if (!g) return;
  for (int i = 0; i < PKV_GRAPH_MAX_BUCKETS; ++i)
    if (g->exec[i]) cudaGraphExecDestroy(g->exec[i]);
  delete g;
}

}  // extern "C"
