"""Plain data of the library's configuration: the flag and format constants
of include/kvq.h and Python mirrors of kvq_fmt / kvq_config.

Nothing here loads libkvq.so, so the seeded workload generators (and through
them the CPU oracle's timed runs) can use these shapes without the CUDA
library.  The ctypes marshalling of a Config lives in kvq.py.
"""

from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

AXIS_TOKEN = 0
AXIS_CHANNEL = 1
ROTATE_K = 1
ROTATE_V = 2
K_PRE_ROPE = 4
TBQ4_K = 8
TBQ4_V = 16
ZP_K = 32
ZP_V = 64
DT_F16 = 0
DT_BF16 = 1

DEV_CAPACITY = 1
DEV_PAGE = 2
DEV_RANGE = 4
DEV_LENGTH = 8
DEV_STALL = 16
DEV_BOUNDS = 32


@dataclass(frozen=True)
class Fmt:
    bits: int
    group: int
    axis: int = AXIS_TOKEN


@dataclass
class Config:
    """Mirror of kvq_config."""

    L: int
    H_kv: int
    H_q: int
    D: int
    batch: int
    max_T: int
    in_dtype: int = DT_F16
    k_fmt: Fmt = Fmt(4, 32)
    v_fmt: Fmt = Fmt(4, 32)
    k_cold: Optional[Fmt] = None
    v_cold: Optional[Fmt] = None
    hot_window: int = 0
    residual_window: int = 0
    flags: int = 0
    rope_theta: float = 10000.0
    sign_seed: int = 0
    page_tokens: int = 0
    n_pages: int = 0
    max_pages_per_seq: int = 0
