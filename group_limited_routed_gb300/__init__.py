"""Beam MoE layer (group-limited routed experts) for GB300 / sm_103a.

The compute path is the C-ABI library ``libbeam_moe.so`` (hand-written CUDA);
this package only marshals arguments to it.  ``inputs`` draws seeded synthetic
workloads.  Importing the package does not load the library; the first call
of an entry point does, and fails loudly when it is missing.
"""
from .config import BeamMoEConfig  # noqa: F401


def __getattr__(name):
    # the binding is loaded lazily so that the input generator can be imported
    # on machines without the compiled library
    if name in ("route", "select", "forward", "forward_routed", "workspace_size", "Workspace",
                "check_status", "BeamError", "library_path", "lib", "set_stage_events",
                "set_debug", "layout", "kernels_per_forward", "EXPORTS", "forward_noalloc",
                "forward_nvfp4", "pack_scales", "Fp4Weight", "NVFP4", "ep_dispatch",
                "ep_experts", "ep_combine", "EpWorkspace", "forward_boundary",
                "forward_nvfp4_a16", "NVFP4_A16", "ep_experts_nvfp4", "forward_fp8",
                "Fp8Weight", "FP8", "fp8_quantize_rows", "ep_experts_fp8", "BF16",
                "forward_mxfp8", "Mxfp8Weight", "MXFP8"):
        from . import api
        return getattr(api, name)
    raise AttributeError(name)
