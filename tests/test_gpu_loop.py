"""GPU parity over whole decode loops, and checkpoint/resume of a loop.

Loops (64 steps, the cosine schedule, full refresh every 3 steps, per-step drift
N(0, 0.05) of the fresh Q/K/V):
  * MAR-L shape: batch 128 doubled to 256, 16 heads, d = 64, 320 tokens, top-32 refresh,
    in both forms of the cached layer (one launch reading the active rows in place, and
    gather + cache-aware attention);
  * 512 px shape: batch 64 doubled to 128, 16 heads, d = 80, 32x32 + 64 = 1088 tokens,
    top-64 refresh (up to 25 + 25 + 64 active tokens);
  * MAR-H shape at a reduced batch: 32 doubled to 64, 16 heads, d = 80, 320 tokens,
    top-64 refresh.

The GPU runs the whole batch through ``DecodeStep``; the oracle follows sampled rows with
its own cache (rows are independent). After every step: outputs within the bf16
tolerance, refresh sets exact (a near-tie within 1e-6 relative is logged and the GPU row
then takes the oracle's set so the two stay comparable), and the sampled rows of the GPU
cache bit-identical to the oracle's.

Checkpoint/resume: the MAR-L loop's state (the layer-3 cache and the drift streams) is
saved at step 30, every tensor is dropped, the state is restored into fresh tensors and
the loop continues; every later step's output and the final cache are bit-identical to
those of the uninterrupted run (the library keeps no state between calls).
"""
import hashlib
import io

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

LOOPS = {
    "mar_l": workloads.CONFIGS["mar_l_loop"],
    "px512": workloads.CONFIGS["px512"],
    "mar_h": workloads.CONFIGS["mar_h"].scaled(B=32, K=64, G=0, J=0, steps=64),
}


def _schedule(cfg):
    """Per-image generation orders and per-step generating positions (host)."""
    sched = workloads.cosine_schedule(cfg.n_img, cfg.steps)
    orders = [workloads.generation_order(cfg.n_img, cfg.n_buf, cfg.seed * 1000 + b) for b in range(cfg.B)]
    gens = []
    for t in range(cfg.steps):
        g = torch.stack([workloads.gen_positions(o, sched, t) for o in orders]).to(torch.int32)
        gens.append(torch.cat([g, g], 0) if cfg.cfg else g)   # cond/uncond rows share positions
    return sched, gens


def _streams(cfg, dev):
    shape = (cfg.Bp, cfg.H, cfg.N, cfg.d)
    return [workloads.DriftStream(shape, cfg.seed * 10_000 + 97 * i, torch.bfloat16, dev, cfg.drift)
            for i in range(6)]


@pytest.mark.parametrize("name,fused_gather", [("mar_l", True), ("mar_l", False), ("px512", True),
                                               ("mar_h", True)])
def test_decode_loop(name, fused_gather):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    cfg = LOOPS[name]
    dev = torch.device("cuda")
    sched, gens = _schedule(cfg)
    assert sum(sched) == cfg.n_img and min(sched) >= 1
    streams = _streams(cfg, dev)
    shape = (cfg.Bp, cfg.H, cfg.N, cfg.d)
    Kc = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
    Vc = torch.zeros_like(Kc)
    a_max = 2 * max(sched) + cfg.K
    step = DecodeStep(cfg.Bp, cfg.H, cfg.N, cfg.d, cfg.K, a_max, device=dev, max_gen=max(sched),
                      fused_gather=fused_gather)
    rows = [0, cfg.B, cfg.Bp - 1] if name != "px512" else [0, cfg.Bp - 1]
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


def _digest(x: torch.Tensor) -> str:
    return hashlib.sha256(P.bits(x).tobytes()).hexdigest()


def _run(cfg, gens, step, state, t0, t1, dev):
    """Steps t0 .. t1 - 1 of the loop on ``state`` (Kc, Vc, streams); returns per-step output digests."""
    Kc, Vc, streams = state
    out = []
    for t in range(t0, t1):
        Q2, K2, V2, Q3, K3, V3 = (s.advance() for s in streams)
        gen = gens[t].to(dev)
        just = gens[t - 1].to(dev) if t > 0 else gen[:, :0]
        excl = torch.cat([gen, just], 1).contiguous()
        res = step.run(t, (Q2, K2, V2), (Q3, K3, V3), (Kc, Vc), gen, excl)
        out.append((res[0], _digest(res[1])) + ((_digest(res[2]),) if res[0] == "cached" else ()))
    return out


def test_checkpoint_resume_is_bit_identical():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    cfg = LOOPS["mar_l"]
    dev = torch.device("cuda")
    sched, gens = _schedule(cfg)
    a_max = 2 * max(sched) + cfg.K
    step = DecodeStep(cfg.Bp, cfg.H, cfg.N, cfg.d, cfg.K, a_max, device=dev, max_gen=max(sched))
    shape = (cfg.Bp, cfg.H, cfg.N, cfg.d)

    def fresh_state():
        Kc = torch.zeros(shape, dtype=torch.bfloat16, device=dev)
        return Kc, torch.zeros_like(Kc), _streams(cfg, dev)

    # uninterrupted
    st = fresh_state()
    straight = _run(cfg, gens, step, st, 0, cfg.steps, dev)
    final = (_digest(st[0]), _digest(st[1]))
    del st
    # interrupted at step 30: the state goes to bytes, every tensor is dropped
    st = fresh_state()
    first = _run(cfg, gens, step, st, 0, 30, dev)
    buf = io.BytesIO()
    torch.save({"Kc": st[0].cpu(), "Vc": st[1].cpu(), "next_step": 30,
                "streams": [(s.x.cpu(), s.step) for s in st[2]]}, buf)
    del st
    torch.cuda.empty_cache()
    buf.seek(0)
    ck = torch.load(buf)
    streams = _streams(cfg, dev)
    for s, (x, k) in zip(streams, ck["streams"]):
        s.x.copy_(x.to(dev))
        s.step = k
    restored = (ck["Kc"].to(dev), ck["Vc"].to(dev), streams)
    rest = _run(cfg, gens, step, restored, ck["next_step"], cfg.steps, dev)
    assert first + rest == straight
    assert (_digest(restored[0]), _digest(restored[1])) == final
    assert mar.mar_status_read(step.status) == 0
