"""Multi-tenant decode step of the Llama-3-8B-shape stack replayed from one CUDA graph.

The serving loop of the page's "Architecture de service" section -- a request
names its variant, the variant's delta is applied to the one resident base and
the forward pass runs -- over two full layers of the stack (q 4096x4096, k/v
1024x4096, o 4096x4096, gate/up 14336x4096, down 4096x14336).  Each variant of
each matrix is a fine-tuned W_ft = bf16(W_base + Laplace(0, b_v)) compressed by
bd_compress_batch; its bits must equal the oracle's and its alpha agree within
1e-6.  The 14 multi-tenant linears (64 tokens, ids over four variants with one
variant left without tokens) are captured in one CUDA graph with the
workspaces shared by matrices of one shape, exactly as the benchmark's stack
step does, replayed twice, and checked element by element on sampled outputs
against the oracle's multi-tenant linear (fed the oracle's own bits and alpha).
"""
import numpy as np
import pytest
import torch

import oracle
from bit_delta_tenant_gb300 import bitdelta as bd
from bit_delta_tenant_gb300 import synth, workloads
from helpers import ALPHA_REL, assert_y_close, sample_outputs, y_host

pytestmark = pytest.mark.gpu

N_VAR = 4
EMPTY = 2          # a variant with no tokens
SCALES = [5e-4, 1e-3, 1.5e-3, 2e-3]
M = 64


def _compress_variants(w_base, seed):
    """GPU bits/alpha of every variant (one bd_compress_batch call) and the oracle's."""
    n_out, n_in = w_base.shape
    wb_h = synth.as_u16(w_base)
    fts, outs = [], []
    for v in range(N_VAR):
        g = synth.generator(seed * 17 + v, "cuda")
        d = synth.laplace_f32((n_out, n_in), SCALES[v], g, "cuda")
        fts.append((w_base.float() + d).to(torch.bfloat16))
        del d
        outs.append((torch.empty((n_out, n_in // 8), dtype=torch.uint8, device="cuda"),
                     torch.empty((1,), dtype=torch.float32, device="cuda")))
    descs = bd.compress_descs([(w_base, wf, 0, b, a) for wf, (b, a) in zip(fts, outs)])
    ws = torch.empty((bd.bd_compress_batch_workspace_size(descs),), dtype=torch.uint8, device="cuda")
    bd.bd_compress_batch(descs, ws)
    torch.cuda.synchronize()
    ref = []
    for v, wf in enumerate(fts):
        b_h, a32, a64 = oracle.compress(wb_h, synth.as_u16(wf), 0)
        assert np.array_equal(outs[v][0].cpu().numpy(), b_h), f"variant {v}: packed bits differ from the oracle"
        got = float(outs[v][1].item())
        assert abs(got - a64[0]) <= ALPHA_REL * abs(a64[0]), f"variant {v}: alpha {got} vs {a64[0]}"
        ref.append((b_h, a32))
    del fts
    return outs, ref


def test_two_layer_multi_tenant_decode_graph_matches_oracle():
    c = workloads.LLAMA3_8B_STACK
    rng = np.random.default_rng(5)
    live = [v for v in range(N_VAR) if v != EMPTY]
    ids_h = rng.choice(live, size=M).astype(np.int32)
    ids_h[:len(live)] = live                       # every live variant has at least one token
    ids = torch.from_numpy(ids_h).to("cuda")
    mats, xs, wss = [], {}, {}
    for layer in range(2):
        for j, (name, n_out, n_in) in enumerate(c["matrices"]):
            seed = workloads.matrix_seed(c["seed"], 7000 + 10 * layer + j)
            w_base = synth.bf16_normal((n_out, n_in), c["sigma"], synth.generator(seed, "cuda"), "cuda")
            outs, ref = _compress_variants(w_base, seed)
            if n_in not in xs:
                xs[n_in] = synth.activations(M, n_in, 30_000 + n_in, "cuda")
            if (n_out, n_in) not in wss:   # matrices of one shape share a workspace, as in the benchmark
                wss[(n_out, n_in)] = torch.empty((bd.bd_linear_grouped_workspace_size(M, N_VAR, n_out, n_in),),
                                                 dtype=torch.uint8, device="cuda")
            y = torch.full((M, n_out), float("nan"), dtype=torch.bfloat16, device="cuda")
            mats.append(dict(name=f"L{layer}.{name}", w_base=w_base, outs=outs, ref=ref, y=y,
                             x=xs[n_in], ws=wss[(n_out, n_in)]))
    modes = [0] * N_VAR

    def step():
        for mt in mats:
            bd.bd_linear_grouped(mt["x"], ids, mt["w_base"], [b for b, _ in mt["outs"]],
                                 [a for _, a in mt["outs"]], modes, mt["y"], mt["ws"])

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        step()                                     # eager pass (kernel attributes, device info)
    torch.cuda.synchronize()
    for mt in mats:
        mt["y"].fill_(float("nan"))
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    g.replay()
    torch.cuda.synchronize()
    assert bd.bd_get_device_status() == bd.BD_OK
    first = [mt["y"].clone() for mt in mats]
    for mt in mats:
        mt["y"].fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert bd.bd_get_device_status() == bd.BD_OK
    x_h = {k: synth.as_u16(v) for k, v in xs.items()}
    for i, mt in enumerate(mats):
        assert torch.equal(first[i], mt["y"]), f"{mt['name']}: the two replays differ"
        n_out, n_in = mt["w_base"].shape
        ts, js = sample_outputs(M, n_out, 200, seed=i)
        y_ref, mag = oracle.linear_grouped_sampled(x_h[n_in], ids_h, synth.as_u16(mt["w_base"]),
                                                   [b for b, _ in mt["ref"]], [a for _, a in mt["ref"]],
                                                   np.array(modes, np.int32), ts, js)
        assert_y_close(y_host(mt["y"])[ts, js], y_ref, mag, mt["name"])
