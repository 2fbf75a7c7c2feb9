"""Shared helpers of the GPU layer tests: run the CUDA layer through the C
ABI, run the oracle on chosen tokens, and compare the two."""
from __future__ import annotations

import numpy as np
import torch

from mixture_experts_layer_100_b300 import synth
from oracle import moe_oracle as om

DEV = "cuda"
TOL = {"f32": 1e-5, "bf16": 2e-2, "e4m3": 6e-2, "e4m3_ue8m0": 6e-2}


class LazyStack:
    """[n, ...] device tensor whose items are fetched to the host as float64
    one at a time (keeps the V3-sized weights off the host)."""

    def __init__(self, t: torch.Tensor):
        self.t = t
        self.shape = tuple(t.shape)

    def __getitem__(self, i):
        return self.t[int(i)].double().cpu().numpy()


def host(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy()


def device_weights(w: synth.Weights):
    return {k: getattr(w, k).to(DEV).contiguous() for k in ("w_router", "w13", "w2", "ws13", "ws2")}


def run_layer(p: synth.Preset, wd: dict, xd: torch.Tensor, bd: torch.Tensor, gamma: float = 0.0, ws=None,
              out_dtype=None):
    from mixture_experts_layer_100_b300 import binding as B
    cfg = B.config_from_preset(p)
    ws = B.alloc_workspace(cfg) if ws is None else ws
    dt = out_dtype or synth.torch_dtype(p.dtype)
    out = torch.full((p.T, p.d), float("nan"), dtype=dt, device=DEV)
    idx = torch.empty((p.T, p.K), dtype=torch.int32, device=DEV)
    gate = torch.empty((p.T, p.K), dtype=torch.float32, device=DEV)
    counts = torch.empty((p.E,), dtype=torch.int32, device=DEV)
    mom = torch.empty(1, dtype=torch.float32, device=DEV)
    B.moe_layer_forward(cfg, xd, B.make_weights(**wd), bd, gamma, out, idx, gate, counts, mom, ws)
    torch.cuda.synchronize()
    code = B.moe_device_error(ws)
    assert code == 0, hex(code)
    return {"out": out, "topk_idx": idx, "topk_gate": gate, "counts": counts, "max_over_mean": mom, "ws": ws}


def oracle_rows(p, w: synth.Weights, x: torch.Tensor, b: torch.Tensor, tokens=None):
    """Oracle layer output for the given tokens (all when None)."""
    xs = x if tokens is None else x[torch.as_tensor(tokens)]
    lazy = w.w13.is_cuda
    W = (lambda t: LazyStack(t)) if lazy else (lambda t: t.double().numpy())
    return om.layer_forward(host(xs).astype(np.float64), host(w.w_router), W(w.w13), W(w.w2), W(w.ws13),
                            W(w.ws2), b.cpu().numpy(), p.G, p.K, p.M, p.group_topk)


def near_tie(scores, bias, G, K, M, gk, eps=2e-5):
    """True when the oracle's own group or expert choice for this token is
    decided by a margin below eps (so that fp32 rounding of the scores may
    legitimately flip it)."""
    sp = om.biased_scores(scores[None, :], bias)
    gs = np.sort(om.group_scores(sp, G, gk)[0])[::-1]
    if M < G and gs[M - 1] - gs[M] < eps:
        return True
    mask = np.repeat(om.select_groups(om.group_scores(sp, G, gk), M)[0], len(bias) // G)
    cand = np.sort(np.where(mask, sp[0], -np.inf))[::-1]
    return cand[K - 1] - cand[K] < eps


def compare(p, res, ref, bias, tokens=None, dtype=None, max_flip=0.01):
    """Element-wise comparison of the GPU output with the oracle's on the
    tokens whose routing agrees; routing disagreements must be near-ties of
    the oracle's own scores. `bias` is the bias the routing used."""
    dtype = dtype or p.expert_dtype
    toks = np.arange(p.T) if tokens is None else np.asarray(tokens)
    gi = res["topk_idx"].cpu().numpy()[toks]
    same = np.array([set(a) == set(b) for a, b in zip(gi, ref["topk_idx"])])
    bias = np.asarray(bias.cpu() if torch.is_tensor(bias) else bias, np.float32)
    for j in np.nonzero(~same)[0]:
        assert near_tie(ref["scores"][j], bias, p.G, p.K, p.M, p.group_topk), (toks[j], gi[j], ref["topk_idx"][j])
    assert (~same).sum() <= max(1, int(max_flip * len(toks))), (~same).sum()
    got = res["out"].float().cpu().numpy()[toks][same]
    want = ref["out"][same]
    err = np.abs(got - want).max() / np.abs(want).max()
    assert err <= TOL[dtype], err
    return err, int((~same).sum())


def quantize_device_weights(wd: dict, ue8m0: bool = False) -> dict:
    """e4m3 codes + 128x128 block scales of the expert weights, made on the
    GPU by moe_quantize_weights_e4m3 (or its power-of-two variant); the
    router stays in the master dtype."""
    from mixture_experts_layer_100_b300 import binding as B
    quant = B.moe_quantize_weights_e4m3_ue8m0 if ue8m0 else B.moe_quantize_weights_e4m3
    out = {"w_router": wd["w_router"]}
    for k in ("w13", "w2", "ws13", "ws2"):
        w = wd[k]
        n, r, c = w.shape
        q = torch.empty((n, r, c), dtype=torch.uint8, device=DEV)
        sc = torch.empty((n, (r + 127) // 128, (c + 127) // 128), dtype=torch.float32, device=DEV)
        quant(w, q, sc)
        out[k] = q
        out[k + "_scale"] = sc
    torch.cuda.synchronize()
    return out


def oracle_rows_fp8(p, w: synth.Weights, x: torch.Tensor, b: torch.Tensor, tokens=None):
    """FP8 oracle layer output for the given tokens (all when None), with the
    preset's scale rule."""
    xs = x if tokens is None else x[torch.as_tensor(tokens)]
    lazy = w.w13.is_cuda
    W = (lambda t: LazyStack(t)) if lazy else (lambda t: t.double().numpy())
    return om.layer_forward_fp8_full(host(xs).astype(np.float64), host(w.w_router), W(w.w13), W(w.w2),
                                     W(w.ws13), W(w.ws2), b.cpu().numpy(), p.G, p.K, p.M, p.group_topk,
                                     ue8m0=p.expert_dtype == "e4m3_ue8m0")


def oracle_rows_cpp(p, w: synth.Weights, x: torch.Tensor, b: torch.Tensor, tokens=None, expert_dtype=None):
    """The C++ oracle's layer output for the given tokens (all when None),
    streaming one expert's weights at a time to the host (so V3-sized weights
    may stay on the device). expert_dtype: "e4m3" / "e4m3_ue8m0" for the FP8
    path, else the master-precision path."""
    from oracle import cpp
    xs = host(x if tokens is None else x[torch.as_tensor(np.asarray(tokens))])
    n = xs.shape[0]
    s = cpp.router_scores(xs, host(w.w_router))
    idx, gate = cpp.select_experts(s, np.asarray(b.cpu() if torch.is_tensor(b) else b, np.float32), p.G, p.K, p.M,
                                   p.group_topk)
    f8 = expert_dtype in ("e4m3", "e4m3_ue8m0")
    ue = expert_dtype == "e4m3_ue8m0"
    acc = np.zeros((n, p.d), np.float64)
    for j in range(p.S):
        cpp.expert_accumulate(xs, np.arange(n), host(w.ws13[j]), host(w.ws2[j]), None, acc, fp8=f8, ue8m0=ue)
    for e in np.unique(idx):
        rows, slots = np.nonzero(idx == e)
        cpp.expert_accumulate(xs, rows, host(w.w13[int(e)]), host(w.w2[int(e)]), gate[rows, slots], acc, fp8=f8,
                              ue8m0=ue)
    return {"scores": s, "topk_idx": idx, "topk_gate": gate, "out": acc}


def stratified_tokens(topk_idx: np.ndarray, E: int, n: int, seed: int, hot: int = 3) -> np.ndarray:
    """A seeded token sample for the full-size parity tests that reaches every
    expert's first and last permuted row (the first row of its first 128-row
    tile and the last row of its ragged tail), the first and last row of every
    tile of the `hot` most loaded experts, and uniform random tokens up to n
    tokens in all. Positions follow the expert-major, token-ascending order of
    the routing given (the layer's own)."""
    from oracle import cpp
    T, K = topk_idx.shape
    st, _ = cpp.permutation(topk_idx, E)
    off = cpp.exclusive_offsets(cpp.expert_counts(topk_idx, E))
    pos = []
    for e in range(E):
        if off[e + 1] > off[e]:
            pos += [off[e], off[e + 1] - 1]
    counts = np.diff(off)
    for e in np.argsort(-counts, kind="stable")[:hot]:
        for p0 in range(off[e], off[e + 1], 128):
            pos += [p0, min(p0 + 127, off[e + 1] - 1)]
    picked = set(int(st[q]) for q in pos)
    rng = np.random.default_rng(seed)
    rest = rng.permutation(T)
    for t in rest:
        if len(picked) >= n:
            break
        picked.add(int(t))
    return np.array(sorted(picked), np.int64)
