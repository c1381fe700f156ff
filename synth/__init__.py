"""Seeded synthetic inputs for the ReplaySSM decode workloads.

This package only draws random numbers and shapes them (activation
functions applied to raw draws, L2 normalisation of keys and queries,
rounding to bfloat16 storage). It holds none of the decode method's
arithmetic, so both the CUDA path and the CPU oracle can consume its output
without sharing any of the computation under test.
"""

from .inputs import (  # noqa: F401
    DeltaWorkload,
    Mamba2Workload,
    accept_counts,
    bf16_round,
    delta_initial_state,
    delta_step_inputs,
    mamba2_draft_inputs,
    mamba2_initial_state,
    mamba2_params,
    mamba2_step_inputs,
    spec_draft_inputs,
)
