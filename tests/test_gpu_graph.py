"""GEMM calls captured in a CUDA graph and replayed.

A sequence of calls -- the CTA-pair kernel (FP16 TN, TF32), the FP32 SIMT
kernels (split-K in clusters and the TMA-fed one), split-K in clusters on
the tensor cores, the single-CTA kernel and the workspace path --
is captured once on a side stream after one eager warm-up call of each (the
library's per-device caches are filled outside the capture), then replayed.
Every replay must give exactly the eager results: the kernels are
deterministic and the graph holds the same launches.
"""
import pytest
import torch

from tests import parity

pytestmark = pytest.mark.gpu


def _problems():
    out = []
    for path, (M, N, K), seed in (("f16_tn", (1024, 2048, 512), 1), ("tf32", (768, 1536, 1000), 2),
                                  ("f32", (300, 520, 1000), 3), ("f16_tn", (100, 1000, 2048), 4),
                                  ("bf16_nn", (129, 260, 72), 5), ("f32", (2176, 2304, 96), 7)):
        A, B, C = parity.host_operands(path, M, N, K, seed=seed)
        out.append((path, A.cuda(), B.cuda(), C.cuda()))
    return out


def test_graph_replay_matches_eager():
    import dense_gemm_09_gb300 as dg
    probs = _problems()
    # the workspace path: odd pitches, both operands copied
    A, B, C = parity.host_operands("tf32", 129, 257, 301, seed=6)
    wsA, wsB, wsC = A.cuda(), B.cuda(), C.cuda()
    ws = torch.empty(dg.tf32_workspace_bytes(wsA, wsB), dtype=torch.uint8, device="cuda")

    def run_all(outs):
        for (path, dA, dB, C0), out in zip(probs, outs[:-1]):
            out.copy_(C0)
            parity.fn(path)(dA, dB, out, 1.25, 0.5)
        outs[-1].copy_(wsC)
        dg.gemm_tf32_ws(wsA, wsB, outs[-1], 1.25, 0.5, workspace=ws)

    eager = [torch.empty_like(p[3]) for p in probs] + [torch.empty_like(wsC)]
    run_all(eager)  # also fills the library's per-device caches
    torch.cuda.synchronize()
    graph_out = [torch.empty_like(e) for e in eager]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run_all(graph_out)
    for _ in range(3):
        for t in graph_out:
            t.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert dg.device_status(clear=False) == dg.OK
        for e, t in zip(eager, graph_out):
            assert torch.equal(e, t)
