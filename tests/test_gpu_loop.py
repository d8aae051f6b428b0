"""GPU parity over a whole decode loop: MAR-L shape (batch 128 doubled to 256, 16 heads,
d=64, 320 tokens), 64 steps with the cosine schedule, top-32 refresh, full refresh every
3 steps and per-step drift N(0, 0.05) of the fresh Q/K/V.

The GPU runs the whole batch through ``DecodeStep``; the oracle follows three sampled
rows with its own cache (rows are independent). After every step: outputs within the
bf16 tolerance, refresh sets exact (a near-tie within 1e-6 relative is logged and the
GPU row then takes the oracle's set so the two stay comparable), and the sampled rows of
the GPU cache bit-identical to the oracle's.
"""
import numpy as np
import pytest
import torch

import _parity as P
import cache_aware_attention_gb300 as mar
import oracle
import workloads
from cache_aware_attention_gb300.step import DecodeStep, is_full_refresh
from oracle.loop import OracleRows

pytestmark = pytest.mark.gpu


def _schedule(cfg):
    """Per-image generation orders and per-step generating positions (host)."""
    sched = workloads.cosine_schedule(cfg.n_img, cfg.steps)
    orders = [workloads.generation_order(cfg.n_img, cfg.n_buf, cfg.seed * 1000 + b) for b in range(cfg.B)]
    gens = []
    for t in range(cfg.steps):
        g = torch.stack([workloads.gen_positions(o, sched, t) for o in orders]).to(torch.int32)
        gens.append(torch.cat([g, g], 0) if cfg.cfg else g)   # cond/uncond rows share positions
    return sched, gens


@pytest.mark.parametrize("fused_gather", [True, False])
def test_decode_loop_mar_l(fused_gather):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    cfg = workloads.CONFIGS["mar_l_loop"]
    dev = torch.device("cuda")
    sched, gens = _schedule(cfg)
    assert sum(sched) == cfg.n_img and min(sched) >= 1
    shape = (cfg.Bp, cfg.H, cfg.N, cfg.d)
    streams = [workloads.DriftStream(shape, cfg.seed * 10_000 + 97 * i, torch.bfloat16, dev, cfg.drift)
               for i in range(6)]
    Kc = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
    Vc = torch.zeros_like(Kc)
    a_max = 2 * max(sched) + cfg.K
    step = DecodeStep(cfg.Bp, cfg.H, cfg.N, cfg.d, cfg.K, a_max, device=dev, max_gen=max(sched),
                      fused_gather=fused_gather)
    rows = [0, cfg.B, cfg.Bp - 1]
    orc = OracleRows(rows, cfg.K)
    ties, checked = [], 0
    for t in range(cfg.steps):
        Q2, K2, V2, Q3, K3, V3 = (s.advance() for s in streams)
        sl = lambda x: x[rows].cpu()
        gen = gens[t]
        just = gens[t - 1] if t > 0 else gen[:, :0]
        excl = torch.cat([gen, just], 1).contiguous()
        if is_full_refresh(t):
            kind, O3 = step.run(t, (Q2, K2, V2), (Q3, K3, V3), (Kc, Vc), gen.to(dev), excl.to(dev))
            ref = orc.step(t, (sl(Q2), sl(K2), sl(V2)), (sl(Q3), sl(K3), sl(V3)), gen[rows].numpy(),
                           excl[rows].numpy())
            assert kind == "full"
            P.assert_close(O3[rows], ref["O"], "bf16", f"step {t} full O")
        else:
            A = excl.shape[1] + cfg.K
            gen_d, excl_d = gen.to(dev), excl.to(dev)
            act = step.active(A)
            mar.mar_attn_full(Q2, K2, V2, step.O2, gen_idx=gen_d, score_out=step.score,
                              workspace=step.workspace, status=step.status)
            mar.mar_refresh_topk(step.score, excl_d, cfg.K, out_idx=step.R, active_out=act,
                                 status=step.status)
            score_rows = step.score[rows].cpu().numpy().astype(np.float64)
            R_rows = step.R[rows].cpu().numpy()
            ref = orc.step(t, (sl(Q2), sl(K2), sl(V2)), (sl(Q3), sl(K3), sl(V3)), gen[rows].numpy(),
                           excl[rows].numpy())
            rel = np.abs(score_rows - ref["score"]) / ref["score"]
            assert rel.max() < 1e-6, f"step {t}: score rel error {rel.max():.3g}"
            tie = P.topk_mismatches(R_rows, ref["R"], ref["score"], excl[rows].numpy(), cfg.K)
            if tie:
                ties += [(t,) + x for x in tie]
                for i, b in enumerate(rows):    # follow the oracle's choice on this row
                    act[b].copy_(torch.from_numpy(ref["active"][i]).to(dev))
            kind, OA, act2 = step.cached_layer(A, (Q3, K3, V3), (Kc, Vc))
            assert np.array_equal(act2[rows].cpu().numpy(), ref["active"])
            P.assert_close(OA[rows], ref["O"], "bf16", f"step {t} O_A")
        assert np.array_equal(oracle._rows_as_bytes(Kc[rows].cpu()), orc.Kc), f"step {t}: K cache"
        assert np.array_equal(oracle._rows_as_bytes(Vc[rows].cpu()), orc.Vc), f"step {t}: V cache"
        checked += 1
    assert mar.mar_status_read(step.status) == 0
    assert checked == cfg.steps
    if ties:
        print(f"near-ties followed: {ties}")
