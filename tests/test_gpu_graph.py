"""The bucketed CUDA-graph decode executor ("mini-llm-inference-engine" README: CUDA Graph
multi-bucket capture) on the GPU.  A graph launch must produce exactly what the same calls
made directly at the bucket's batch size produce (same kernels, same plans): outputs and
caches compared bit for bit, several layers of different KV formats, padding rows inert,
two consecutive steps through one executor, the fused step with rotation; and the outputs
match the FP64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_09_gb300 import pkv, runner
from paged_kv_attention_09_gb300 import workloads as W

from gpu_util import TOL, max_err

pytestmark = pytest.mark.gpu

BUCKETS = [1, 2, 4, 8]
LENS = [37, 16, 1, 70, 100, 17, 64, 33]  # one step's context lengths for B_max = 8
FORMATS = [W.F32, W.INT8, W.FP8, W.BF16]  # one layer each


def layer_workloads(seed):
    # the same seed draws the same tables and values; each layer stores them in its format
    return [W.small_workload(seed, num_q_heads=8, num_kv_heads=2, head_dim=64, kv_dtype=kv,
                             q_dtype=W.F32, new_dtype=W.F32, decode_lens=LENS)
            for kv in FORMATS]


class Step:
    """Device buffers of one decode step for B_max sequences over several layers."""

    def __init__(self, wls, n):
        b = wls[0].batches[0]
        self.wls, self.n = wls, n
        self.dws = [runner.upload(wl, "cuda") for wl in wls]  # history rows appended
        rows = wls[0].step_rows[:b.num_seqs]
        dev = torch.device("cuda")
        self.bt = torch.from_numpy(b.block_tables).to(dev)
        lens = b.context_lens.copy()
        lens[n:] = 0
        slots = wls[0].slots[rows].astype(np.int32).copy()
        slots[n:] = -1
        self.lens = torch.from_numpy(lens).to(dev)
        self.slots = torch.from_numpy(slots).to(dev)
        self.pos = torch.from_numpy((b.context_lens - 1).astype(np.int32)).to(dev)
        self.k = [dw.k_src[torch.from_numpy(rows).to(dev)].contiguous() for dw in self.dws]
        self.v = [dw.v_src[torch.from_numpy(rows).to(dev)].contiguous() for dw in self.dws]
        self.q = [dw.batches[0].q for dw in self.dws]
        self.out = [torch.full_like(dw.batches[0].out, 7.0) for dw in self.dws]
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)

    def layers(self):
        return [pkv.GraphLayer(dw.cache, q, o, k, v)
                for dw, q, o, k, v in zip(self.dws, self.q, self.out, self.k, self.v)]


def direct(step, B, fused, ws, rope):
    for dw, q, o, k, v in zip(step.dws, step.q, step.out, step.k, step.v):
        if fused:
            pkv.pkv_decode_step(dw.cache, q[:B], k[:B], v[:B], step.slots[:B],
                                step.pos[:B] if rope else None, 1.0e4, step.bt[:B], step.lens[:B],
                                dw.wl.scale, o[:B], ws, step.status)
        else:
            pkv.pkv_append(dw.cache, k[:B], v[:B], step.slots[:B], step.status)
            pkv.pkv_decode_attn(dw.cache, q[:B], step.bt[:B], step.lens[:B], dw.wl.scale, o[:B],
                                ws, step.status)


def own_workspace(graph):
    """A separate zero-filled workspace of the executor's size (None when it needs none)."""
    w = graph.workspace
    return None if w is None else torch.zeros_like(w)


def same_bytes(a, b):
    return torch.equal(a.view(torch.uint8), b.view(torch.uint8))


@pytest.mark.parametrize("fused,rope", [(False, False), (True, False), (True, True)])
@pytest.mark.parametrize("n", [1, 3, 5, 8])
def test_graph_equals_direct_calls_and_oracle(n, fused, rope):
    g_step = Step(layer_workloads(9100), n)
    d_step = Step(layer_workloads(9100), n)
    graph = pkv.DecodeGraph(g_step.layers(), g_step.bt, g_step.lens, g_step.wls[0].scale, BUCKETS,
                            slot_mapping=g_step.slots, fused=fused,
                            positions=g_step.pos if rope else None, rope_theta=1.0e4,
                            dev_status=g_step.status)
    B = graph.bucket(n)
    assert B == min(b for b in BUCKETS if b >= n)
    graph.launch(n)
    direct(d_step, B, fused, own_workspace(graph), rope)
    torch.cuda.synchronize()
    assert int(g_step.status.item()) == 0 and int(d_step.status.item()) == 0
    for gd, dd, go, do in zip(g_step.dws, d_step.dws, g_step.out, d_step.out):
        assert same_bytes(go[:B], do[:B])
        assert same_bytes(gd.cache.k, dd.cache.k) and same_bytes(gd.cache.v, dd.cache.v)
        if gd.cache.k_scale is not None:
            assert torch.equal(gd.cache.k_scale, dd.cache.k_scale)
        assert torch.all(go[n:B] == 0)   # padding rows: zero output
        assert torch.all(go[B:] == 7.0)  # rows past the bucket: untouched
    # against the oracle: the step of the first n sequences
    for wl, go in zip(g_step.wls, g_step.out):
        b = wl.batches[0]
        rows = wl.step_rows[:n]
        oc = oracle.cache_from_workload(wl, rows=wl.history_rows)
        if fused:
            ref = oracle.decode_step(oc, b.q[:n], b.q_dtype, wl.k_src[rows], wl.v_src[rows],
                                     wl.new_dtype, wl.slots[rows],
                                     (b.context_lens[:n] - 1).astype(np.int32) if rope else None,
                                     1.0e4, b.block_tables[:n], b.context_lens[:n], wl.scale)
        else:
            oracle.append(oc, wl.k_src[rows], wl.v_src[rows], wl.new_dtype, wl.slots[rows])
            ref = oracle.decode(oc, b.q[:n], b.q_dtype, b.block_tables[:n], b.context_lens[:n],
                                wl.scale)
        assert max_err(go[:n].cpu().numpy().astype(np.float64), ref) <= TOL[wl.kv_dtype]
    graph.close()


def test_graph_two_steps_with_new_contents():
    """The executor replays over whatever the buffers hold: a second step with other
    queries, one more token per sequence and new slots gives the direct calls' result."""
    g_step = Step(layer_workloads(9200), 6)
    d_step = Step(layer_workloads(9200), 6)
    graph = pkv.DecodeGraph(g_step.layers(), g_step.bt, g_step.lens, g_step.wls[0].scale, BUCKETS,
                            slot_mapping=g_step.slots, dev_status=g_step.status)
    ws = own_workspace(graph)
    graph.launch(6)
    direct(d_step, 8, False, ws, False)
    # next step: the 6 live sequences overwrite their newest token's slot with new rows and
    # get new queries (the buffers are rewritten in place)
    for st in (g_step, d_step):
        gen = torch.Generator(device="cuda").manual_seed(5)
        for q, k, v in zip(st.q, st.k, st.v):
            q.copy_(torch.randn(q.shape, device="cuda", generator=gen))
            k.copy_(torch.randn(k.shape, device="cuda", generator=gen))
            v.copy_(torch.randn(v.shape, device="cuda", generator=gen))
    graph.launch(6)
    direct(d_step, 8, False, ws, False)
    torch.cuda.synchronize()
    for gd, dd, go, do in zip(g_step.dws, d_step.dws, g_step.out, d_step.out):
        assert same_bytes(go, do)
        assert same_bytes(gd.cache.k, dd.cache.k) and same_bytes(gd.cache.v, dd.cache.v)
    graph.close()


def test_graph_launch_bounds():
    st = Step(layer_workloads(9300), 2)
    graph = pkv.DecodeGraph(st.layers()[:1], st.bt, st.lens, st.wls[0].scale, [2, 4],
                            slot_mapping=st.slots)
    assert [graph.bucket(n) for n in (0, 1, 2, 3, 4, 5)] == [0, 2, 2, 4, 4, 0]
    graph.launch(0)  # no-op
    with pytest.raises(pkv.PkvError):
        graph.launch(5)
    torch.cuda.synchronize()
    graph.close()
