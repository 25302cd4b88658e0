"""Runs one layer call of every expert format at several batch sizes on the
bounds-checked build and prints `format T status` per call.  Started by
test_gpu_checked_build.py in a process of its own with
BEAM_MOE_DEVICE_CHECKS=1 (the variable selects the checked library when the
package is imported)."""
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import group_limited_routed_gb300 as pkg  # noqa: E402
from group_limited_routed_gb300 import api, inputs  # noqa: E402

# 16: decode-sized 16-row blocks; 40 and 64: 256-row blocks on CTA pairs, the
# last expert's block at most half full (a pair half with no valid row);
# 200: several token blocks per expert; 1100 (128 experts): the
# counting-sort permutation and the tensor-core router
SIZES = {"bf16": [16, 40, 64, 200, 1100], "fp8": [16, 40, 64, 200, 1100],
         "mxfp8": [16, 40, 64, 200], "nvfp4": [16, 40, 64, 200], "a16": [16, 40, 64, 200]}


def _cuda(v):
    if isinstance(v, dict):
        return {k: _cuda(x) for k, x in v.items()}
    return v.cuda() if isinstance(v, torch.Tensor) else v


def main():
    assert api._LIB_PATH.endswith(os.path.join("_build_checked", "libbeam_moe.so")), api._LIB_PATH
    for fmt, sizes in SIZES.items():
        wf = "nvfp4" if fmt == "a16" else fmt
        for T in sizes:
            cfg = inputs.CONFIGS["tiny"].replace(T=T, weight_fmt=wf, cpu_generator=True, seed=7 + T,
                                                 n_experts=128 if T > 1000 else 64)
            t = {k: _cuda(v) for k, v in inputs.generate(cfg, "cpu").items()}
            head = (cfg, t["hidden"], t["router_w"], t["corr_bias"])
            if fmt == "bf16":
                ws = pkg.Workspace(cfg, T)
                pkg.forward(*head, t["w_gate"], t["w_up"], t["w_down"], ws=ws)
            elif fmt == "fp8":
                ws = pkg.Workspace(cfg, T, weight_fmt=pkg.FP8)
                pkg.forward_fp8(*head, *[pkg.Fp8Weight.of(t[n]) for n in ("w_gate", "w_up", "w_down")],
                                ws=ws)
            elif fmt == "mxfp8":
                ws = pkg.Workspace(cfg, T, weight_fmt=pkg.MXFP8)
                pkg.forward_mxfp8(*head,
                                  *[pkg.Mxfp8Weight.of(t[n]) for n in ("w_gate", "w_up", "w_down")],
                                  ws=ws)
            else:
                ws = pkg.Workspace(cfg, T, weight_fmt=pkg.NVFP4 if fmt == "nvfp4" else pkg.NVFP4_A16)
                fwd = pkg.forward_nvfp4 if fmt == "nvfp4" else pkg.forward_nvfp4_a16
                fwd(*head, *[pkg.Fp4Weight.of(t[n]) for n in ("w_gate", "w_up", "w_down")], ws=ws)
            print(fmt, T, pkg.check_status(ws), flush=True)


if __name__ == "__main__":
    main()
