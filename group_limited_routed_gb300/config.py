"""Layer shape record passed across the C ABI (mirrors beam_moe_config_t)."""
import ctypes
from dataclasses import dataclass


@dataclass(frozen=True)
class BeamMoEConfig:
    d: int = 5120
    n_experts: int = 256
    n_groups: int = 8
    topk_groups: int = 4
    topk: int = 8
    d_ff: int = 2560
    routed_scale: float = 2.5

    @classmethod
    def of(cls, c) -> "BeamMoEConfig":
        return cls(d=c.d, n_experts=c.n_experts, n_groups=c.n_groups,
                   topk_groups=c.topk_groups, topk=c.topk, d_ff=c.d_ff,
                   routed_scale=c.routed_scale)


class CConfig(ctypes.Structure):
    _fields_ = [("d", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("n_groups", ctypes.c_int32), ("topk_groups", ctypes.c_int32),
                ("topk", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("routed_scale", ctypes.c_float)]

    @classmethod
    def of(cls, c) -> "CConfig":
        return cls(c.d, c.n_experts, c.n_groups, c.topk_groups, c.topk, c.d_ff,
                   float(c.routed_scale))
