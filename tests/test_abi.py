"""The C ABI: the library builds, loads and exports every declared symbol, the
ctypes structs match the C layout, and host-side validation rejects bad
arguments before anything is enqueued (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")


def declared_functions():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", txt)))


def test_every_declared_symbol_is_exported(kda_lib):
    names = declared_functions()
    assert "kda_prefill" in names and "kda_decode_step" in names and "kda_gate_norm" in names
    for n in names:
        assert hasattr(kda_lib, n), f"{n} declared in kda.h but not exported"
    import serving_kda_chunked_gated_gb300.kda as kda
    assert sorted(kda.EXPORTED) == sorted(set(kda.EXPORTED) & set(names))


def test_struct_layout_matches_c(tmp_path):
    import serving_kda_chunked_gated_gb300.kda as kda
    structs = [("kda_prefill_args", kda.PrefillArgs), ("kda_decode_args", kda.DecodeArgs),
               ("kda_short_conv_args", kda.ShortConvArgs), ("kda_short_conv_step_args", kda.ShortConvStepArgs)]
    prog = tmp_path / "layout.c"
    lines = ['#include <stdio.h>', '#include <stddef.h>', f'#include "{HEADER}"', "int main(void){"]
    for cname, py in structs:
        lines.append(f'printf("%zu\\n", sizeof({cname}));')
        lines += [f'printf("%zu\\n", offsetof({cname}, {f[0]}));' for f in py._fields_]
    lines += ["return 0;}"]
    prog.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", str(prog), "-o", str(exe)], check=True)
    out = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()]
    i = 0
    for cname, py in structs:
        assert out[i] == ctypes.sizeof(py), cname
        i += 1
        for f in py._fields_:
            assert out[i] == getattr(py, f[0]).offset, (cname, f[0])
            i += 1


FAKE = 0x7f0000000000  # never dereferenced: validation fails before any launch


def _args(kda, **kw):
    a = kda.PrefillArgs()
    a.num_seqs, a.T_total, a.H, a.dk, a.dv, a.qkv_dtype = 1, 64, 2, 128, 128, kda.KDA_BF16
    cu = np.array([0, 64], dtype=np.int32)
    a.cu_seqlens = FAKE
    a.cu_seqlens_host = cu.ctypes.data
    for name in ("q", "k", "v", "z", "beta", "A", "o"):
        setattr(a, name, FAKE)
    a.g_min, a.scale, a.qk_l2norm, a.norm_eps = -5.0, 1.0, 1, 1e-6
    for key, val in kw.items():
        setattr(a, key, val)
    return a, cu


@pytest.mark.parametrize("mutate,expect", [
    (dict(q=None), 1), (dict(A=None), 1), (dict(cu_seqlens=None), 1),
    (dict(dk=96, dv=96), 2), (dict(dk=128, dv=64), 2), (dict(H=0), 2),
    (dict(qkv_dtype=5), 3), (dict(q=FAKE + 4), 4), (dict(o=FAKE + 8), 4),
    (dict(T_total=65), 5), (dict(g_in=FAKE), 1),
    (dict(S_snap=FAKE, snap_interval=0), 2), (dict(S_snap=FAKE, snap_interval=96), 2),
    (dict(S_snap=FAKE + 4, snap_interval=64), 4),
])
def test_prefill_validation(kda_lib, mutate, expect):
    import serving_kda_chunked_gated_gb300.kda as kda
    a, cu = _args(kda, **mutate)
    assert kda_lib.kda_prefill(ctypes.byref(a), None) == expect
    assert kda_lib.kda_prefill_recurrent(ctypes.byref(a), None) == expect


def test_prefill_seqlens_validation(kda_lib):
    import serving_kda_chunked_gated_gb300.kda as kda
    a, _ = _args(kda)
    bad = np.array([0, 40, 30, 64], dtype=np.int32)
    a.num_seqs, a.cu_seqlens_host = 3, bad.ctypes.data
    assert kda_lib.kda_prefill(ctypes.byref(a), None) == 5
    bad2 = np.array([1, 64], dtype=np.int32)
    a.num_seqs, a.cu_seqlens_host = 1, bad2.ctypes.data
    assert kda_lib.kda_prefill(ctypes.byref(a), None) == 5
    # f32 gate input is not accepted
    a2, _c = _args(kda, g_in=FAKE, y=FAKE, qkv_dtype=kda.KDA_F32)
    assert kda_lib.kda_prefill(ctypes.byref(a2), None) == 3
    assert kda_lib.kda_prefill_workspace_size(ctypes.byref(a2)) == 0


def test_snapshot_count(kda_lib):
    """Rows of the prefix-cache snapshot output: whole intervals per sequence."""
    import serving_kda_chunked_gated_gb300.kda as kda
    cu = np.array([0, 0, 130, 150, 343, 407], dtype=np.int32)
    a, _ = _args(kda, num_seqs=5, T_total=407, cu_seqlens_host=cu.ctypes.data,
                 S_snap=FAKE, snap_interval=64)
    assert kda_lib.kda_prefill_snapshot_count(ctypes.byref(a)) == 2 + 0 + 3 + 1
    a.snap_interval = 128
    assert kda_lib.kda_prefill_snapshot_count(ctypes.byref(a)) == 1 + 0 + 1 + 0
    assert kda.snapshot_count(cu, 128) == 2 and kda.snapshot_count(cu, 64) == 6
    a.snap_interval = 100                                   # not a multiple of the chunk
    assert kda_lib.kda_prefill_snapshot_count(ctypes.byref(a)) == 0
    a.snap_interval, a.S_snap = 64, None                    # snapshots off
    assert kda_lib.kda_prefill_snapshot_count(ctypes.byref(a)) == 0


def test_decode_and_gate_norm_validation(kda_lib):
    import serving_kda_chunked_gated_gb300.kda as kda
    d = kda.DecodeArgs()
    d.N, d.H, d.dk, d.dv, d.num_slots = 4, 2, 128, 128, 4
    for name in ("q", "k", "v", "z", "beta", "A", "state", "o"):
        setattr(d, name, FAKE)
    d2 = kda.DecodeArgs.from_buffer_copy(d)
    d2.o = None
    assert kda_lib.kda_decode_step(ctypes.byref(d2), None) == 1      # neither o nor y
    d3 = kda.DecodeArgs.from_buffer_copy(d)
    d3.dk = d3.dv = 64
    assert kda_lib.kda_decode_step(ctypes.byref(d3), None) == 2
    d4 = kda.DecodeArgs.from_buffer_copy(d)
    d4.num_slots = 3                                                 # no slots, fewer rows than N
    assert kda_lib.kda_decode_step(ctypes.byref(d4), None) == 2
    d5 = kda.DecodeArgs.from_buffer_copy(d)
    d5.state = FAKE + 12
    assert kda_lib.kda_decode_step(ctypes.byref(d5), None) == 4
    d6 = kda.DecodeArgs.from_buffer_copy(d)
    d6.g_in = FAKE                                                  # g_in without y
    assert kda_lib.kda_decode_step(ctypes.byref(d6), None) == 1
    f = kda_lib.kda_gate_norm
    f.argtypes = [ctypes.c_void_p] * 3 + [ctypes.c_float, ctypes.c_void_p, ctypes.c_long,
                                          ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    assert f(FAKE, FAKE, None, 1e-6, FAKE, 10, 96, 0, None) == 2
    assert f(FAKE, FAKE, None, 1e-6, FAKE, 10, 128, 9, None) == 3
    assert f(None, FAKE, None, 1e-6, FAKE, 10, 128, 0, None) == 1
    assert f(FAKE + 2, FAKE, None, 1e-6, FAKE, 10, 128, 0, None) == 4


def test_short_conv_validation(kda_lib):
    import serving_kda_chunked_gated_gb300.kda as kda
    cu = np.array([0, 64], dtype=np.int32)
    a = kda.ShortConvArgs()
    a.num_seqs, a.T_total, a.channels, a.width, a.dtype = 1, 64, 256, 4, kda.KDA_BF16
    a.cu_seqlens, a.cu_seqlens_host = FAKE, cu.ctypes.data
    a.x, a.weight, a.y, a.activation = FAKE, FAKE + 4096, FAKE + 8192, 1
    f = kda_lib.kda_short_conv
    for field, val, expect in (("width", 9, 2), ("width", 0, 2), ("channels", 100, 2), ("dtype", 7, 3),
                               ("y", FAKE, 2), ("x", FAKE + 8, 4), ("T_total", 65, 5), ("weight", None, 1)):
        b = kda.ShortConvArgs.from_buffer_copy(a)
        setattr(b, field, val)
        assert f(ctypes.byref(b), None) == expect, (field, val)
    st = kda.ShortConvStepArgs()
    st.N, st.channels, st.width, st.num_slots, st.dtype = 4, 256, 4, 2, kda.KDA_BF16
    st.x, st.weight, st.y, st.state = FAKE, FAKE, FAKE, FAKE
    assert kda_lib.kda_short_conv_step(ctypes.byref(st), None) == 2     # fewer state rows than tokens
    st.num_slots, st.state = 4, None
    assert kda_lib.kda_short_conv_step(ctypes.byref(st), None) == 1     # width > 1 needs a state


def test_status_strings(kda_lib):
    kda_lib.kda_status_str.restype = ctypes.c_char_p
    assert kda_lib.kda_status_str(0) == b"ok"
    assert b"cu_seqlens" in kda_lib.kda_status_str(5)
    kda_lib.kda_version.restype = ctypes.c_char_p
    assert b"sm_103a" in kda_lib.kda_version()


def test_records_and_scan_validation(kda_lib):
    """kda_prefill_records / kda_prefill_scan: kda_prefill's argument checks,
    then the chunk-parallel workspace, the flags and the schedule's inputs."""
    import serving_kda_chunked_gated_gb300.kda as kda
    a, cu = _args(kda)
    need = kda_lib.kda_prefill_workspace_size(ctypes.byref(a))
    assert need > 256
    for mutate, expect in ((dict(q=None), 1), (dict(T_total=65), 5), (dict(dk=96, dv=96), 2),
                           (dict(o=FAKE + 8), 4)):
        b, _c = _args(kda, **mutate)
        assert kda_lib.kda_prefill_records(ctypes.byref(b), None) == expect
        assert kda_lib.kda_prefill_scan(ctypes.byref(b), 0, None) == expect
    assert kda_lib.kda_prefill_records(ctypes.byref(a), None) == 8          # no workspace
    a.workspace, a.workspace_bytes = FAKE, need - 1
    assert kda_lib.kda_prefill_scan(ctypes.byref(a), 0, None) == 8         # smaller than the records
    a.workspace, a.workspace_bytes = FAKE + 8, need
    assert kda_lib.kda_prefill_records(ctypes.byref(a), None) == 4         # misaligned
    a.workspace = FAKE
    assert kda_lib.kda_prefill_scan(ctypes.byref(a), 2, None) == 2         # unknown flag
    f, _c2 = _args(kda, qkv_dtype=kda.KDA_F32, workspace=FAKE, workspace_bytes=1 << 40)
    assert kda_lib.kda_prefill_records(ctypes.byref(f), None) == 6         # no chunk-parallel schedule
    assert kda_lib.kda_prefill_scan(ctypes.byref(f), kda.SCAN_ZERO_V, None) == 6


def test_prefill_from_host_validation(kda_lib):
    """kda_prefill_from_host: one sequence, slabs a positive multiple of 64, no
    snapshots, host inputs and outputs present, caller staging of the size
    kda_prefill_from_host_staging_size gives (checked before anything is
    enqueued)."""
    import serving_kda_chunked_gated_gb300.kda as kda
    a, _cu = _args(kda, T_total=1000, S_T=FAKE)
    need = kda_lib.kda_prefill_from_host_staging_size(ctypes.byref(a), 256)
    assert need > 2 * 256 * 2 * 128 * (3 * 2 + 4)            # two slabs of q, k, v (bf16) and z at least
    assert kda_lib.kda_prefill_from_host_staging_size(ctypes.byref(a), 100) == 0
    bigger = kda_lib.kda_prefill_from_host_staging_size(ctypes.byref(a), 512)
    assert bigger > need
    call = lambda b, slab=256, st=FAKE, n=need: kda_lib.kda_prefill_from_host(ctypes.byref(b), slab, st, n, None)
    assert call(a, slab=0) == 2 and call(a, slab=100) == 2
    assert call(_args(kda, T_total=1000, S_T=FAKE, num_seqs=2)[0]) == 2
    assert call(_args(kda, T_total=1000, S_T=FAKE, S_snap=FAKE, snap_interval=64)[0]) == 6
    assert call(_args(kda, T_total=1000, S_T=FAKE, q=None)[0]) == 1
    assert call(_args(kda, T_total=1000)[0]) == 1                   # no S_T
    assert call(_args(kda, T_total=1000, S_T=FAKE, g_in=FAKE)[0]) == 1   # g_in without y
    assert call(a, st=None) == 8 and call(a, st=FAKE + 8) == 4 and call(a, n=need - 1) == 8


def test_record_size_per_chunk_head(kda_lib):
    """The chunk-parallel workspace holds one record per (chunk, head): the A
    tile [-W ; Gamma Q - P Gamma K] (128 x 128 fp16), [U ; U_o] (128 x 128
    fp32), (K gamma_C / Gamma)^T (128 x 64 fp16), gamma_C (128 fp32) and the
    64 output rows' scale factors (fp32) -- 115456 bytes, the 112.75 KiB per
    chunk and head that kda.h states; a ragged last chunk takes a whole one."""
    import serving_kda_chunked_gated_gb300.kda as kda
    rec = 128 * 128 * 2 + 128 * 128 * 4 + 128 * 64 * 2 + (128 + 64) * 4
    assert rec == 115456 and rec / 1024 == 112.75
    sizes, keep = [], []
    for T in (64 * 10, 64 * 11, 64 * 11 - 5):
        cu = np.array([0, T], dtype=np.int32)
        keep.append(cu)
        a, _ = _args(kda, T_total=T, H=3)
        a.cu_seqlens_host = cu.ctypes.data
        sizes.append(kda_lib.kda_prefill_workspace_size(ctypes.byref(a)))
    assert sizes[1] - sizes[0] == 3 * rec
    assert sizes[2] == sizes[1]
