"""Layer calls enqueued back to back on one stream, without a host
synchronisation between them, give the outputs of the same calls run one at
a time, bit for bit.  The later kernels of a call are launched with
programmatic stream serialization (a kernel may start while the one before
it still runs and waits on the device for what it reads), so this checks the
ordering between calls: calls of every expert format in a row, and two calls
that share one workspace with different inputs (the second call's kernels
overwrite the buffers the first one's read)."""
import pytest
import torch

import group_limited_routed_gb300 as pkg
from group_limited_routed_gb300 import inputs

pytestmark = pytest.mark.gpu

# (format, T): 16-row blocks with row gather, CTA pairs (T = 64, 300), the
# counting-sort permutation and the separate routing kernels (T = 300)
CASES = [("bf16", 64), ("bf16", 300), ("nvfp4", 16), ("a16", 40), ("fp8", 64), ("mxfp8", 16)]


def _cuda(v):
    if isinstance(v, dict):
        return {k: _cuda(x) for k, x in v.items()}
    return v.cuda() if isinstance(v, torch.Tensor) else v


def _layer(fmt, T, seed):
    """A callable that runs the layer of one format into its own output,
    and its workspace."""
    wf = "nvfp4" if fmt == "a16" else fmt
    cfg = inputs.CONFIGS["tiny"].replace(T=T, weight_fmt=wf, cpu_generator=True, seed=seed)
    t = {k: _cuda(v) for k, v in inputs.generate(cfg, "cpu").items()}
    if fmt == "bf16":
        ws = pkg.Workspace(cfg, T)
        w, fwd = (t["w_gate"], t["w_up"], t["w_down"]), pkg.forward
    elif fmt == "fp8":
        ws = pkg.Workspace(cfg, T, weight_fmt=pkg.FP8)
        w, fwd = [pkg.Fp8Weight.of(t[n]) for n in ("w_gate", "w_up", "w_down")], pkg.forward_fp8
    elif fmt == "mxfp8":
        ws = pkg.Workspace(cfg, T, weight_fmt=pkg.MXFP8)
        w, fwd = [pkg.Mxfp8Weight.of(t[n]) for n in ("w_gate", "w_up", "w_down")], pkg.forward_mxfp8
    else:
        ws = pkg.Workspace(cfg, T, weight_fmt=pkg.NVFP4 if fmt == "nvfp4" else pkg.NVFP4_A16)
        w = [pkg.Fp4Weight.of(t[n]) for n in ("w_gate", "w_up", "w_down")]
        fwd = pkg.forward_nvfp4 if fmt == "nvfp4" else pkg.forward_nvfp4_a16

    def call(x, out, ws=ws):
        fwd(cfg, x, t["router_w"], t["corr_bias"], *w, out=out, ws=ws,
            stream=torch.cuda.current_stream())

    return cfg, t["hidden"], call, ws


def _bits(x):
    return x.view(torch.int16)


def test_calls_of_every_format_back_to_back_match_single_calls():
    layers = [_layer(fmt, T, 50 + i) for i, (fmt, T) in enumerate(CASES)]
    ref = []
    for cfg, x, call, ws in layers:
        out = torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16, device="cuda")
        call(x, out)
        torch.cuda.synchronize()
        assert pkg.check_status(ws) == 0
        ref.append(out.clone())
    outs = [torch.full_like(r, float("nan")) for r in ref]
    for order in (range(len(layers)), reversed(range(len(layers)))):
        for o in outs:
            o.fill_(float("nan"))
        for i in order:                     # no synchronisation in between
            layers[i][2](layers[i][1], outs[i])
        torch.cuda.synchronize()
        for i, (o, r) in enumerate(zip(outs, ref)):
            assert torch.equal(_bits(o), _bits(r)), CASES[i]
    for cfg, x, call, ws in layers:
        assert pkg.check_status(ws) == 0


@pytest.mark.parametrize("fmt,T", [("bf16", 64), ("nvfp4", 16), ("fp8", 64)])
def test_two_calls_sharing_a_workspace_match_single_calls(fmt, T):
    cfg, x1, call, ws = _layer(fmt, T, 80)
    x2 = inputs.generate(cfg.replace(seed=81), "cpu", weights=False)["hidden"].cuda()
    o1 = torch.empty(T, cfg.d, dtype=torch.bfloat16, device="cuda")
    o2 = torch.empty_like(o1)
    call(x1, o1)
    torch.cuda.synchronize()
    r1 = o1.clone()
    call(x2, o2)
    torch.cuda.synchronize()
    r2 = o2.clone()
    for _ in range(3):
        o1.fill_(float("nan"))
        o2.fill_(float("nan"))
        call(x1, o1)                        # the second call reuses the workspace at once
        call(x2, o2)
        call(x1, o1)
        torch.cuda.synchronize()
        assert torch.equal(_bits(o1), _bits(r1)) and torch.equal(_bits(o2), _bits(r2))
    assert pkg.check_status(ws) == 0
