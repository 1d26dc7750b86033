"""CPU oracle (test infrastructure only): fp64 numpy compile/link and a brute-force twin.

Only tests, the smoke check and the benchmark's CPU-baseline leg import this package.
"""
from .pic_oracle import (OracleModel, OracleStore, OutOfBlocks, LinkMeta, LinkOut, SeqJob,  # noqa: F401
                         run_jobs, full_prefill, compile_chunks, rms_norm, rope, rope_inv_freq,
                         causal_attention, silu)
