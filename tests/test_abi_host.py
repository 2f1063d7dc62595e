"""Host-side checks of the C-ABI library (no GPU): it loads, it exports every entry point
include/cc.h declares, and its host helpers (position ids) agree bit for bit with the
oracle."""
import os
import re

import numpy as np
import pytest

from conftest import ROOT
from oracle import decoder as O
from synth.configs import layer_fp32_T128, pair_T2048, stack28_T8192, varlen_T32768, ImageSpan

import cohere_compass_decoder_gb300._lib as L


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(L.LIB_PATH):
        from cohere_compass_decoder_gb300.build import build
        build()
    return L.lib()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "cc.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cc_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert len(names) >= 16
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(L.EXPORTS) == names


def test_status_strings(lib):
    assert L.status_string(0) == "ok"
    assert "invalid" in L.status_string(1)


def _spans(wl):
    return [(i.seq, i.start, i.grid_t, i.grid_h, i.grid_w) for i in wl.images]


@pytest.mark.parametrize("make", [layer_fp32_T128, pair_T2048, stack28_T8192, varlen_T32768])
def test_positions_bit_exact_on_workloads(lib, make):
    wl = make()
    pos, delta = L.cc_build_mrope_positions(_spans(wl), wl.seq_lens)
    want, wdelta = O.positions(wl.seq_lens, _spans(wl))
    assert np.array_equal(np.asarray(pos, dtype=np.int64), want)
    assert delta == wdelta.tolist()


def test_positions_bit_exact_random_layouts(lib):
    rng = np.random.default_rng(123)
    for _ in range(50):
        n_seqs = int(rng.integers(1, 4))
        lens, spans = [], []
        for s in range(n_seqs):
            L_ = int(rng.integers(0, 200))
            lens.append(L_)
            k = 0
            while True:
                k += int(rng.integers(0, 20))
                t, h, w = int(rng.integers(1, 3)), int(rng.integers(1, 6)), int(rng.integers(1, 6))
                if k + t * h * w > L_:
                    break
                spans.append((s, k, t, h, w))
                k += t * h * w
        rng.shuffle(spans)
        pos, delta = L.cc_build_mrope_positions(spans, lens)
        want, wdelta = O.positions(lens, spans)
        assert np.array_equal(np.asarray(pos, dtype=np.int64).reshape(3, -1), want.reshape(3, -1))
        assert delta == wdelta.tolist()


@pytest.mark.parametrize("bad", [
    [(0, 10, 1, 2, 2)],          # runs past the end of the 12-token sequence
    [(1, 0, 1, 1, 1)],           # no sequence 1
    [(0, 0, 1, 2, 2), (0, 3, 1, 1, 1)],   # overlapping images
    [(0, 0, 0, 1, 1)],           # empty grid
    [(0, -1, 1, 1, 1)],
])
def test_positions_reject_bad_spans(lib, bad):
    with pytest.raises(L.CCError) as e:
        L.cc_build_mrope_positions(bad, [12])
    assert e.value.status == L.CC_ERR_INVALID_ARG


def test_decode_positions(lib):
    pos = L.cc_build_decode_positions([4096, 7, 0], [-12, 0, 3])
    want = O.decode_positions([4096, 7, 0], [-12, 0, 3])
    assert np.array_equal(np.asarray(pos), want)
    with pytest.raises(L.CCError):
        L.cc_build_decode_positions([5], [-9])


def test_struct_layouts_match_header(tmp_path):
    """The ctypes structs mirror the C structs: sizes and field offsets as the C compiler
    lays them out from include/cc.h."""
    import ctypes as C
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    structs = {"cc_model_config": L.cc_model_config, "cc_layer_weights": L.cc_layer_weights,
               "cc_kv_pool": L.cc_kv_pool, "cc_image_span": L.cc_image_span}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "cc.h"', "int main(void){"]
    for name, st in structs.items():
        lines.append(f'printf("{name} %zu\\n", sizeof({name}));')
        for fname, _ in st._fields_:
            lines.append(f'printf("{name}.{fname} %zu\\n", offsetof({name}, {fname}));')
    lines.append("return 0;}")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    out = dict(l.rsplit(" ", 1) for l in subprocess.run([str(exe)], capture_output=True, text=True,
                                                        check=True).stdout.split("\n") if l)
    for name, st in structs.items():
        assert int(out[name]) == C.sizeof(st), name
        for fname, _ in st._fields_:
            assert int(out[f"{name}.{fname}"]) == getattr(st, fname).offset, (name, fname)


# ------------------------------------------------------------ host-side checks of the next rows
def test_q4_tiled_bytes(lib):
    """Blocks of 128 rows x 128 K, 9216 bytes each; an odd number of 64-K groups rounds up."""
    assert lib.cc_q4_tiled_bytes(128, 128) == 9216
    assert lib.cc_q4_tiled_bytes(256, 2048) == 2 * 16 * 9216
    assert lib.cc_q4_tiled_bytes(19456, 2048) == 152 * 16 * 9216
    assert lib.cc_q4_tiled_bytes(2048, 10240) == 16 * 80 * 9216
    assert lib.cc_q4_tiled_bytes(128, 192) == 2 * 9216          # 3 groups -> 2 blocks
    for rows, k in [(100, 128), (128, 100), (0, 64), (128, 0), (-128, 64)]:
        assert lib.cc_q4_tiled_bytes(rows, k) == 0


def test_q4_entry_points_reject_bad_arguments_before_any_device_work(lib):
    dummy = 256      # never dereferenced: the checks come first
    assert lib.cc_pack_q4_tiles(dummy, dummy, dummy, 100, 128, dummy, None) == L.CC_ERR_UNSUPPORTED
    assert lib.cc_pack_q4_tiles(dummy, dummy, dummy, 128, 96, dummy, None) == L.CC_ERR_UNSUPPORTED
    assert lib.cc_pack_q4_tiles(None, dummy, dummy, 128, 128, dummy, None) == L.CC_ERR_INVALID_ARG
    assert lib.cc_pack_q4_tiles(dummy, dummy, dummy, 0, 128, dummy, None) == L.CC_OK
    assert lib.cc_op_gemm_q4(dummy, dummy, dummy, 129, 128, 64, 1.0, 0, None) == L.CC_ERR_UNSUPPORTED
    assert lib.cc_op_gemm_q4(dummy, dummy, dummy, 64, 100, 64, 1.0, 0, None) == L.CC_ERR_UNSUPPORTED
    assert lib.cc_op_gemm_q4(None, dummy, dummy, 64, 128, 64, 1.0, 0, None) == L.CC_ERR_INVALID_ARG
    assert lib.cc_op_gemm_q4(dummy, dummy, dummy, 0, 128, 64, 1.0, 0, None) == L.CC_OK
    assert lib.cc_layer_plan_attach_q4(None, None, None) == L.CC_ERR_INVALID_ARG
    assert lib.cc_decode_step_q4(None, None, None, None, None, 0, 0, None, None) == L.CC_ERR_INVALID_ARG
    assert lib.cc_logits_q4(None, None, None, 0, None, None) == L.CC_ERR_INVALID_ARG


def test_mrope_layout_argument_is_checked(lib):
    section = L._i32_array((24, 20, 20))
    for layout in (2, -1):
        assert lib.cc_op_mrope_table_layout(256, 4, 128, 5e4, section, layout, 256, None) == \
            L.CC_ERR_INVALID_ARG
    bad = L._i32_array((24, 20, 21))   # does not sum to head_dim / 2
    assert lib.cc_op_mrope_table_layout(256, 4, 128, 5e4, bad, 1, 256, None) == L.CC_ERR_INVALID_ARG
    assert lib.cc_op_mrope_table_layout(256, 0, 128, 5e4, section, 1, 256, None) == L.CC_OK


def test_layernorm_widths_are_checked_before_any_device_work(lib):
    """Every multiple of 128 up to 4096 is a supported row width; others are refused on the
    host (the pointers below are never dereferenced)."""
    dummy = 256
    for H in (100, 4224, 8192):
        assert lib.cc_op_layernorm(dummy, dummy, dummy, 4, H, 1e-5, None, None) == \
            L.CC_ERR_UNSUPPORTED
    assert lib.cc_op_layernorm(dummy, dummy, dummy, 0, 4096, 1e-5, None, None) == L.CC_OK
    assert lib.cc_op_layernorm(dummy, dummy, dummy, 4, 0, 1e-5, None, None) == L.CC_ERR_INVALID_ARG
