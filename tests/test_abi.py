"""Host-side checks of the C ABI (no GPU needed): the library loads, exports every entry
point that include/spd.h declares, and validates arguments / sizes the workspace on the
host."""
import ctypes as C
import os
import re

import pytest

from speculative_pipeline_decoding_spd_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "spd.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(spd_[a-z_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(B.LIB_PATH):
        from speculative_pipeline_decoding_spd_gb300 import build
        build.build()
    return B.load()


def test_header_declares_the_abi():
    names = declared_functions()
    for must in ("spd_create", "spd_prefill", "spd_step", "spd_generate", "spd_get_trace", "spd_destroy"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert sorted(n for n, _, _ in B.SIGNATURES) == declared_functions()


def test_struct_layouts_match_the_c_compiler(tmp_path):
    """Every field offset and struct size of the ctypes mirror equals what a C compiler
    computes from include/spd.h."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    structs = [B.spd_dims, B.spd_layer_weights, B.spd_target_weights, B.spd_pdm_weights, B.spd_config,
               B.spd_stats, B.spd_trace_rec, B.spd_trace_view]
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "spd.h"', 'int main(void){']
    for st in structs:
        lines.append(f'printf("%zu\\n", sizeof({st.__name__}));')
        for f, _ in st._fields_:
            lines.append(f'printf("%zu\\n", offsetof({st.__name__}, {f}));')
    lines.append("return 0;}")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    want = []
    for st in structs:
        want.append(C.sizeof(st))
        want += [getattr(st, f).offset for f, _ in st._fields_]
    assert got == want


def _dims(**kw):
    base = dict(L=36, d=2560, Hq=32, Hkv=8, hd=128, F=9728, V=151936, rope_theta=1e4, rms_eps=1e-6, dtype=B.SPD_BF16)
    base.update(kw)
    return B.spd_dims(*[base[k] for k, _ in B.spd_dims._fields_])


def _cfg(n=8, anchors=(0, 9, 18, 27, 35), max_seq=1100, max_new=512, T=0.0, force_p=-1.0):
    a = (C.c_int32 * 8)(*anchors)
    return B.spd_config(n, len(anchors), a, T, 2, max_seq, max_new, force_p, None, 0, 1, 0)


def test_workspace_bytes_on_host(lib):
    pw = B.spd_pdm_weights(4, None, None, None, None)
    nb = B.spd_workspace_bytes(_dims(), pw, _cfg())
    # KV: 36 layers x 1100 positions x 8 heads x 128 x bf16 x (K, V) plus 4 draft layers
    kv = 2 * (36 + 4) * 1100 * 8 * 128 * 2
    assert kv < nb < kv + 400e6
    assert B.spd_workspace_bytes(_dims(), pw, _cfg(max_seq=5000)) > nb


@pytest.mark.parametrize("kw,cfgkw", [
    (dict(Hq=30), {}),                       # Hq % Hkv != 0
    (dict(hd=96), {}),                       # unsupported head dim
    (dict(dtype=7), {}),
    ({}, dict(n=0)),
    ({}, dict(n=37)),                        # n > L
    ({}, dict(anchors=(1, 9))),              # first anchor must be the embedding
    ({}, dict(anchors=(0, 9, 9))),           # strictly increasing
    ({}, dict(anchors=(0, 40))),             # beyond L
    ({}, dict(max_seq=100)),                 # max_seq < max_new + n + 1
    ({}, dict(force_p=1.5)),
    ({}, dict(force_p=0.5, T=1.0)),          # forced drafts are a greedy test mode
])
def test_invalid_arguments_are_rejected(lib, kw, cfgkw):
    pw = B.spd_pdm_weights(4, None, None, None, None)
    with pytest.raises(B.SPDError) as e:
        B.spd_workspace_bytes(_dims(**kw), pw, _cfg(**cfgkw))
    assert e.value.code == B.SPD_EINVAL
    assert B.spd_last_error(None)


def test_create_rejects_null_weights_without_touching_the_device(lib):
    tw = B.spd_target_weights(None, None, None, None)
    with pytest.raises(B.SPDError) as e:
        B.spd_create(_dims(), tw, None, _cfg(), 0, 0, 0)
    assert e.value.code == B.SPD_EINVAL
