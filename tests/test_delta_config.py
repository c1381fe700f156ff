"""The delta kernels' launch configuration, read from the library on the CPU.

``replayssm_delta_kernel_config`` reports, for given sizes, the block layout
the GDN/KDA decode and verify kernels launch with: prep warps and their
depth, state stages, the vector slots between prep and consumers, consumer
groups and warps, rows per unit. No GPU is needed. These tests hold every
configuration the library picks over a grid of sizes to the pipeline's
ownership rules and to the shared-memory and thread limits, run the picked
slot and stage counts through the barrier-protocol simulation of
``test_pipeline_protocol``, and pin the configurations of the b256 layers
that the measurements quote.
"""

import ctypes
import itertools

import pytest

from recurrent_state_fp32_b300 import _abi, api
from test_pipeline_protocol import run_slots, run_stages

B300_SMEM = 232448


def raw(kind, dk, dv, W, K, read_copy, in_dtype="bf16", smem=0):
    d = _abi.Dims({"gdn": _abi.GDN, "kda": _abi.KDA, "mamba2": _abi.MAMBA2}[kind], 256, 32, 1,
                  dk, dv, W, _abi.BF16 if in_dtype == "bf16" else _abi.F32)
    out = _abi.DeltaConfig()
    rc = _abi.lib.replayssm_delta_kernel_config(ctypes.byref(d), K, int(read_copy), smem,
                                                ctypes.byref(out))
    return rc, {n: int(getattr(out, n)) for n, _ in _abi.DeltaConfig._fields_}


def grid():
    for kind, dk, dv, W, K, rc, ind in itertools.product(
            ("gdn", "kda"), (64, 128), range(32, 257, 32), (1, 5, 16, 64), (1, 2, 4, 8),
            (True, False), ("bf16", "f32")):
        if K <= W:
            yield kind, dk, dv, W, K, rc, ind


def test_every_picked_configuration_keeps_the_rules():
    seen_slots, seen_stages, picked = set(), set(), 0
    for kind, dk, dv, W, K, rc_, ind in grid():
        rc, c = raw(kind, dk, dv, W, K, rc_, ind)
        if rc == _abi.ERR_UNSUPPORTED:
            continue
        assert rc == _abi.OK, (kind, dk, dv, W, K, rc_, ind, rc)
        picked += 1
        where = (kind, dk, dv, W, K, rc_, ind, c)
        G, NS, NP = c["consumer_groups"], c["state_stages"], c["prep_warps"]
        assert G == 4 and NS % G == 0 and NS >= 4 and NP >= 1 and c["depth"] >= 1, where
        assert c["rows_per_unit"] * c["units_per_head"] == dv, where
        assert c["rows_per_unit"] % (32 * c["consumer_warps_per_group"]) == 0, where
        assert c["rows_per_unit"] // c["consumer_warps_per_group"] <= 128, where
        assert c["threads"] <= 512 and 0 < c["smem_bytes"] <= B300_SMEM, where
        nsl, nrb = c["vector_slots"], c["units_per_head"]
        if c["tensor_cores"]:
            assert kind == "gdn" and rc_ and ind == "bf16" and K >= 2 and W <= 16, where
            assert nsl == NP * c["depth"] and c["consumer_warps_per_group"] == 2, where
        else:
            assert c["threads"] == 32 * (G * c["consumer_warps_per_group"] + 1 + NP), where
            if not rc_:
                assert NS >= 8 or NP == 1, where  # FP32 tiles want 8 stages
        # every fill of a slot from one warp; every group sees every fill of its slots
        assert nsl % NP == 0 and (nsl * nrb) % G == 0, where
        seen_slots.add((NP, nsl, nrb))
        seen_stages.add(NS)
    assert picked > 300
    for NP, nsl, nrb in sorted(seen_slots):
        for seed in range(12):
            assert run_slots(NP, nsl, nrb, 4, 2 * nsl + 7, seed) == [], (NP, nsl, nrb, seed)
    for NS in sorted(seen_stages):
        for seed in range(12):
            assert run_stages(NS, 4, 60, seed) == [], (NS, seed)


def test_the_measured_layers():
    """b256, d_k = d_v = 128, W = 16, BF16 read copy and inputs."""
    gdn = api.delta_kernel_config(api.LayerDims("gdn", 256, 32, dk=128, dv=128), 1)
    kda = api.delta_kernel_config(api.LayerDims("kda", 256, 32, dk=128, dv=128), 1)
    for c in (gdn, kda):
        assert (c["tensor_cores"], c["prep_warps"], c["depth"], c["consumer_warps_per_group"],
                c["rows_per_unit"], c["vector_slots"], c["threads"]) == (0, 7, 1, 2, 64, 14, 512)
    assert gdn["state_stages"] == 8 and kda["state_stages"] == 4
    # the speculative workload (b512, K = 4) on the tensor cores: 7 x 2 prep
    # stages would need 249,856 bytes of dynamic shared memory, so 6 x 2
    spec = api.delta_kernel_config(api.LayerDims("gdn", 512, 32, dk=128, dv=128), 4)
    assert (spec["tensor_cores"], spec["prep_warps"], spec["depth"], spec["state_stages"]) == \
        (1, 6, 2, 4)
    big = api.delta_kernel_config(api.LayerDims("gdn", 512, 32, dk=128, dv=128), 4,
                                  smem_limit=260000)
    assert (big["prep_warps"], big["depth"], big["smem_bytes"]) == (7, 2, 249856)


def test_tensor_core_switch(monkeypatch):
    dims = api.LayerDims("gdn", 512, 32, dk=128, dv=128)
    monkeypatch.setenv("REPLAYSSM_DELTA_TENSOR_CORES", "0")
    c = api.delta_kernel_config(dims, 4)
    assert c["tensor_cores"] == 0 and c["vector_slots"] % c["prep_warps"] == 0
    monkeypatch.setenv("REPLAYSSM_DELTA_TENSOR_CORES", "1")
    assert api.delta_kernel_config(dims, 4)["tensor_cores"] == 1
    # KDA and the FP32 read path never take the tensor-core kernel
    assert api.delta_kernel_config(api.LayerDims("kda", 512, 32, dk=128, dv=128), 4)["tensor_cores"] == 0
    assert api.delta_kernel_config(dims, 4, read_copy=False)["tensor_cores"] == 0


def test_arguments():
    assert raw("mamba2", 128, 64, 16, 1, True)[0] == _abi.ERR_INVALID_ARG
    assert raw("gdn", 128, 128, 16, 0, True)[0] == _abi.ERR_INVALID_ARG
    assert raw("gdn", 128, 128, 16, 9, True)[0] == _abi.ERR_INVALID_ARG
    assert raw("gdn", 128, 128, 4, 8, True)[0] == _abi.ERR_INVALID_ARG   # K > W
    assert raw("gdn", 128, 128, 16, 1, True, smem=-1)[0] == _abi.ERR_INVALID_ARG
    assert raw("gdn", 96, 128, 16, 1, True)[0] == _abi.ERR_UNSUPPORTED   # d_k not 64 or 128
    assert raw("gdn", 128, 128, 16, 1, True, smem=4096)[0] == _abi.ERR_UNSUPPORTED
    assert raw("gdn", 128, 128, 16, 1, True, smem=B300_SMEM)[1] == raw("gdn", 128, 128, 16, 1, True)[1]
    d = _abi.Dims(_abi.GDN, 1, 1, 1, 128, 128, 16, _abi.BF16)
    assert _abi.lib.replayssm_delta_kernel_config(ctypes.byref(d), 1, 1, 0, None) == _abi.ERR_INVALID_ARG
    assert _abi.lib.replayssm_delta_kernel_config(None, 1, 1, 0, ctypes.byref(_abi.DeltaConfig())) \
        == _abi.ERR_INVALID_ARG
