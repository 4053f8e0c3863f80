"""The C-ABI library loads without a GPU, exports every function that
include/qg.h declares, and the binding's ctypes structs match the header's
layout (checked by compiling a C program against the header)."""
import ctypes
import os
import re
import subprocess

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "qg.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qg_[a-z0-9_]+)\s*\(", text)))


def test_header_and_binding_agree_on_exports():
    import quantized_gemv_gated_gb300 as qg
    assert sorted(qg.EXPORTS) == declared_functions()


def test_library_loads_and_exports_every_declared_symbol():
    import quantized_gemv_gated_gb300 as qg
    L = qg.lib()
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, missing
    out = subprocess.run(["nm", "-D", "--defined-only", qg.library_path()], capture_output=True, text=True).stdout
    for n in declared_functions():
        assert re.search(rf"\bT {n}$", out, flags=re.M), n


def test_host_only_entry_points_without_gpu():
    import quantized_gemv_gated_gb300 as qg
    assert qg.qg_q6k_planar_bytes(13, 512) == 16 * 2 * 210
    assert qg.qg_q6k_planar_bytes(8, 300) == 0
    assert qg.qg_q4k_planar_bytes(13, 512) == 16 * 2 * 144
    assert qg.qg_q4k_planar_bytes(8, 300) == 0
    assert qg.qg_lmhead_argmax_workspace_bytes() == 16
    with pytest.raises(qg.QgError) as e:
        qg.qg_gemv_q4k(0, 0, 0, 4, 256)
    assert e.value.code == qg.QG_ERR_ARG
    with pytest.raises(qg.QgError) as e:
        qg.qg_gemv_q4k(16, 16, 16, 4, 300)
    assert e.value.code == qg.QG_ERR_SHAPE
    with pytest.raises(qg.QgError) as e:
        qg.qg_gemv_q6k(16, 16, 16, 0, 256)
    assert e.value.code == qg.QG_ERR_EMPTY
    assert "empty" in qg.qg_last_error()
    with pytest.raises(qg.QgError) as e:  # raw Q6_K rows: any k multiple of 256, 2-byte aligned rows
        qg.qg_gemv_q6k(16, 16, 16, 4, 300)
    assert e.value.code == qg.QG_ERR_SHAPE
    with pytest.raises(qg.QgError) as e:
        qg.qg_gemv_q6k(17, 16, 16, 4, 256)
    assert e.value.code == qg.QG_ERR_ARG
    with pytest.raises(qg.QgError) as e:
        qg.qg_gemv_q6k_planar(16, 16, 16, 4, 16640)  # past the engine's K limit
    assert e.value.code == qg.QG_ERR_SHAPE


def test_ctypes_structs_match_header_layout(tmp_path):
    import quantized_gemv_gated_gb300 as qg
    exe = str(tmp_path / "abi_layout")
    subprocess.run(["gcc", "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "abi_layout.c"),
                    "-o", exe], check=True)
    got = dict(line.rsplit(" ", 1) for line in subprocess.run([exe], capture_output=True, text=True,
                                                              check=True).stdout.splitlines())
    py = {"qg_config": qg.QgConfig, "qg_qtensor": qg.QgQTensor, "qg_layer_weights": qg.QgLayerWeights,
          "qg_host_weights": qg.QgHostWeights, "qg_stats": qg.QgStats}
    for key, val in got.items():
        if "." in key:
            s, f = key.split(".")
            assert getattr(py[s], f).offset == int(val), key
        else:
            assert ctypes.sizeof(py[key]) == int(val), key


def test_config_rejects_value_heads_straddling_superblocks():
    """head_v_dim must divide 256 (the ssm_out prologue reduces each head's
    sum of squares inside one 256-element super-block): 96 is refused by the
    host-side check before any device work."""
    import dataclasses
    import synth
    import quantized_gemv_gated_gb300 as qg
    cfg = dataclasses.replace(synth.CFG_TINY, name="tiny-dv96", head_v_dim=96, n_v_heads=8)
    w = synth.make_model_weights(cfg)
    with pytest.raises(qg.QgError) as e:
        qg.Model(w)
    assert e.value.code == qg.QG_ERR_SHAPE and "head_v_dim" in qg.qg_last_error()
