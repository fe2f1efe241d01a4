"""Measurements behind the kernels' design choices, as standalone CUDA programs for sm_103a
for sm_103a (built with nvcc into ``probes/_build``):

* ``tc_rate``: clocks per tcgen05.mma for each MMA kind the kernels use or could use (kind::f16,
  kind::f8f6f4, the block-scaled FP4 kinds), for SM pairs and single CTAs, zero and random
  operands, with the SM clock seen while the pipe is busy.
* ``tc_pipeline``: the MXFP4 SM-pair kernel's per-stage structure (commit per stage, producer
  handshake, scale-factor copies into tensor memory) added to back-to-back MMAs one at a time.
* ``tma_stream``: the read rate of a 4096 x 14336 bf16 matrix (the B operand of the skinny
  64 x 14336 x 4096 GEMM) streamed through TMA in column strips, per strip width, box shape,
  ring depth, K split and L2 promotion, with nothing else running, and with each stage held for
  an MMA's time before it is handed back.
* ``host_link``: host <-> device rates between pinned host memory and the GPU for the host-buffer
  entry points (268 MB in, 134 MB out): copy engines on 1, 2 or 4 streams, and kernels that load
  or store pinned host memory directly, per grid size, each direction alone and both at once.

* ``l2_reuse``: how much of a re-read working set (16-192 MB) the L2 still holds after one read, and
  whether what one half of the SMs read is found in L2 by the other half.

``python -m sm_constrained_persistent_gb300.probes`` builds and runs them on cuda:0 and prints
one JSON line per measurement.  Measurement only: nothing here is on the GEMM path.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD = os.path.join(HERE, "_build")
PROBES = ("tc_rate", "tc_pipeline", "tma_stream", "host_link", "l2_reuse")


def build(name: str) -> str:
    """Compiles probe `name` (if stale) and returns the executable's path."""
    src = os.path.join(HERE, f"{name}.cu")
    exe = os.path.join(BUILD, name)
    if os.path.exists(exe) and os.path.getmtime(exe) >= os.path.getmtime(src):
        return exe
    os.makedirs(BUILD, exist_ok=True)
    nvcc = os.environ.get("NVCC", "nvcc")
    tmp = exe + f".tmp{os.getpid()}"
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                    "-o", tmp, src], check=True)
    os.replace(tmp, exe)
    return exe


def run(name: str, timeout: float = 300.0) -> str:
    """Builds and runs probe `name`; returns its output (one JSON object per line)."""
    r = subprocess.run([build(name)], capture_output=True, text=True, timeout=timeout)
    if r.returncode != 0:
        raise RuntimeError(f"probe {name} failed ({r.returncode}): {r.stdout}{r.stderr}")
    return r.stdout
