"""The five synthetic S6 workloads and their input recipes.

Shapes follow the Mamba layer widths the pages mention (Mamba-130M and
Mamba-2.8B model sizes, "Mamba: Linear-Time Sequence Modeling with Selective
State Spaces", experimental setup) and the million-token DNA length (same
page, setup: sequence lengths up to 1M). Value distributions are synthetic:
the pages' datasets (The Pile, PG-19, genomics sets) are stand-ins only.

Notation: Bt = batch, L = sequence length, D = d_inner channels, N = d_state.
"""

from dataclasses import dataclass, field
from typing import Optional


@dataclass(frozen=True)
class ScanWorkload:
    name: str
    batch: int
    seqlen: int
    dim: int
    dstate: int
    in_dtype: str            # "f32" or "bf16": u, delta_raw, z, B, C
    seed: int
    delta_raw_scale: float   # delta_raw ~ scale * N(0, 1)
    a_log_jitter: float      # A_log[d, n] = log(n + 1) + jitter * N(0, 1)
    u_kind: str = "normal"   # "normal" or "alphabet4" (four N(0,1) symbol vectors)
    dt_min: float = 1e-3     # per-channel dt log-uniform in [dt_min, dt_max]
    dt_max: float = 1e-1
    has_z: bool = True
    has_d: bool = True

    @property
    def channels(self) -> int:
        return self.batch * self.dim

    @property
    def channel_tokens(self) -> int:
        return self.batch * self.seqlen * self.dim

    def algorithmic_bytes(self, out_dtype: str) -> int:
        """Bytes that must cross HBM once: read u, delta_raw, z and B, C; write
        y and h_last; read A, D, bias once."""
        s_in = 2 if self.in_dtype == "bf16" else 4
        s_out = 2 if out_dtype == "bf16" else 4
        Bt, L, D, N = self.batch, self.seqlen, self.dim, self.dstate
        n_td = Bt * L * D
        b = n_td * (3 if self.has_z else 2) * s_in      # u, delta_raw (, z)
        b += Bt * L * N * 2 * s_in                      # B, C
        b += n_td * s_out                               # y
        b += Bt * D * N * 4                             # h_last
        b += D * N * 4 + D * 4 * 2                      # A, D, bias
        return b


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    streams: int
    dim: int
    dstate: int
    steps: int
    prefix: ScanWorkload     # scan whose final state initialises h
    in_dtype: str
    seed: int
    delta_raw_scale: float = 1.0

    def algorithmic_bytes_per_step(self, out_dtype: str) -> int:
        """Per decode step: read and write the state h, read u, delta_raw, z,
        B, C, write y. A, D, bias are re-read per step but stay in L2 and are
        counted once per step at their size."""
        s_in = 2 if self.in_dtype == "bf16" else 4
        s_out = 2 if out_dtype == "bf16" else 4
        S, D, N = self.streams, self.dim, self.dstate
        b = 2 * S * D * N * 4                    # h read + write
        b += 3 * S * D * s_in + 2 * S * N * s_in  # u, delta_raw, z, B, C
        b += S * D * s_out                        # y
        b += D * N * 4 + 2 * D * 4                # A, D, bias
        return b


TINY_FP32 = ScanWorkload("tiny_fp32", batch=1, seqlen=512, dim=256, dstate=16, in_dtype="f32",
                         seed=0, delta_raw_scale=0.5, a_log_jitter=0.0)
MAMBA130M_LAYER = ScanWorkload("mamba130m_layer", batch=8, seqlen=2048, dim=1536, dstate=16, in_dtype="bf16",
                               seed=1, delta_raw_scale=0.5, a_log_jitter=0.0)
MAMBA2P8B_LAYER = ScanWorkload("mamba2p8b_layer", batch=4, seqlen=2048, dim=5120, dstate=16, in_dtype="bf16",
                               seed=2, delta_raw_scale=0.5, a_log_jitter=0.1)
DNA_1M = ScanWorkload("dna_1m", batch=1, seqlen=1 << 20, dim=1024, dstate=16, in_dtype="bf16",
                      seed=3, delta_raw_scale=1.0, a_log_jitter=0.0, u_kind="alphabet4")
DECODE256_PREFIX = ScanWorkload("decode256_prefix", batch=256, seqlen=512, dim=5120, dstate=16,
                                in_dtype="bf16", seed=40, delta_raw_scale=0.5, a_log_jitter=0.1)
DECODE256 = DecodeWorkload("decode256", streams=256, dim=5120, dstate=16, steps=1000,
                           prefix=DECODE256_PREFIX, in_dtype="bf16", seed=4, delta_raw_scale=1.0)

CONFIGS = {w.name: w for w in (TINY_FP32, MAMBA130M_LAYER, MAMBA2P8B_LAYER, DNA_1M, DECODE256)}


def get_config(name: str):
    return CONFIGS[name]
