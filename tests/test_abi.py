"""The C-ABI library builds, loads and exports every symbol include/specverify.h declares (CPU).

Only host-side argument checks are exercised here: they return before any CUDA call, so they run
without a GPU.
"""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "specverify.h")


@pytest.fixture(scope="module")
def libpath():
    from speculative_decoding_verification_35_gb300 import _build
    return _build.build()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_ ]*[\s\*]+([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)


def test_header_declares_the_api():
    names = declared_functions()
    assert set(names) == {"spec_verify", "spec_verify_workspace_size", "spec_verify_ex", "spec_verify_range",
                          "spec_verify_noalloc",
                          "spec_verify_commit", "spec_verify_fused", "spec_draft_ngram", "spec_verify_tree",
                          "spec_verify_status_from_bits", "spec_verify_status_string", "spec_verify_host",
                          "spec_shard_stats", "spec_shard_decide", "spec_shard_chunks", "spec_shard_sums",
                          "spec_shard_finish"}


def test_library_exports_every_declared_symbol(libpath):
    out = subprocess.run(["nm", "-D", "--defined-only", libpath], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, name
    L = ctypes.CDLL(libpath)
    for name in declared_functions():
        assert hasattr(L, name)


def test_binding_lists_every_export(libpath):
    from speculative_decoding_verification_35_gb300 import specverify as sv
    assert set(sv.EXPORTS) == set(declared_functions())


def test_header_compiles_as_c(tmp_path):
    c = tmp_path / "t.c"
    c.write_text('#include "specverify.h"\nint main(void){ sv_debug d = {0}; (void)d; return SV_OK; }\n')
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), "-c", str(c),
                           "-o", str(tmp_path / "t.o")])


def test_binding_structs_match_the_header(tmp_path):
    """The ctypes structures of the binding have the C structures' sizes and every field's offset."""
    from speculative_decoding_verification_35_gb300 import specverify as sv
    structs = (("sv_debug", sv.SvDebug), ("sv_device_buffers", sv.SvDeviceBuffers))
    lines = []
    for cname, py in structs:
        lines.append(f'printf("%zu\\n", sizeof({cname}));')
        for field, _ in py._fields_:
            lines.append(f'printf("%zu\\n", offsetof({cname}, {field}));')
    c = tmp_path / "sizes.c"
    c.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "specverify.h"\n'
                 'int main(void){ ' + " ".join(lines) + ' return 0; }\n')
    exe = tmp_path / "sizes"
    subprocess.check_call(["gcc", "-std=c99", "-I", os.path.dirname(HEADER), str(c), "-o", str(exe)])
    got = iter(map(int, subprocess.check_output([str(exe)]).split()))
    for cname, py in structs:
        assert ctypes.sizeof(py) == next(got), cname
        for field, _ in py._fields_:
            assert getattr(py, field).offset == next(got), (cname, field)


def test_host_side_checks_without_gpu(libpath):
    from speculative_decoding_verification_35_gb300 import specverify as sv
    assert sv.spec_verify_workspace_size(64, 128256, 5) > 0
    assert sv.spec_verify_workspace_size(-1, 10, 1) == 0
    assert sv.spec_verify_workspace_size(4, 10, 32) == 0
    fake = 1 << 20  # never dereferenced: every call below fails its host checks first
    args = dict(target_logits=fake, draft_logits=fake, dtype=sv.SV_BF16, draft_tokens=fake, seq_offsets=fake,
                gammas=fake, B=4, V=100, max_gamma=4, temperature=1.0, seed=1, step=0, out_tokens=fake,
                out_num_accepted=fake, device_status=None, workspace=fake, workspace_bytes=1 << 30, debug=None,
                cuda_stream=None)

    def call(**kw):
        a = dict(args); a.update(kw)
        return sv.spec_verify_ex(**a)

    assert call(temperature=-1.0) == sv.SV_ERR_INVALID_ARG
    assert call(temperature=float("nan")) == sv.SV_ERR_INVALID_ARG
    assert call(temperature=float("inf")) == sv.SV_ERR_INVALID_ARG
    assert call(temperature=1e-45) == sv.SV_ERR_INVALID_ARG
    assert call(V=0) == sv.SV_ERR_INVALID_ARG
    assert call(B=-1) == sv.SV_ERR_INVALID_ARG
    assert call(max_gamma=32) == sv.SV_ERR_INVALID_ARG
    assert call(dtype=7) == sv.SV_ERR_INVALID_ARG
    assert call(target_logits=None) == sv.SV_ERR_INVALID_ARG
    # draft_logits NULL at T > 0 is valid (point-mass drafts), but never without draft tokens
    assert call(draft_logits=None, draft_tokens=None) == sv.SV_ERR_INVALID_ARG
    assert call(draft_tokens=None) == sv.SV_ERR_INVALID_ARG
    assert call(target_logits=fake + 1) == sv.SV_ERR_INVALID_ARG
    assert call(workspace=None) == sv.SV_ERR_WORKSPACE
    assert call(workspace_bytes=16) == sv.SV_ERR_WORKSPACE
    assert call(workspace=fake + 64) == sv.SV_ERR_WORKSPACE
    assert call(B=0) == sv.SV_OK  # nothing to do, nothing launched


def test_status_helpers(libpath):
    from speculative_decoding_verification_35_gb300 import specverify as sv
    assert sv.spec_verify_status_from_bits(0) == sv.SV_OK
    assert sv.spec_verify_status_from_bits((1 << 5) | (1 << 3)) == sv.SV_ERR_BAD_TOKEN
    assert sv.spec_verify_status_from_bits((1 << 5) | (1 << 4)) == sv.SV_ERR_BAD_OFFSETS
    assert sv.spec_verify_status_from_bits(1 << 6) == sv.SV_ERR_EMPTY_ROW
    assert sv.spec_verify_status_from_bits(1 << 9) == sv.SV_ERR_CAPACITY
    for code in range(10):
        assert sv.spec_verify_status_string(code).startswith("SV_")


def test_commit_host_side_checks_without_gpu(libpath):
    from speculative_decoding_verification_35_gb300 import specverify as sv
    fake = 1 << 20  # never dereferenced: every call below returns before any CUDA call
    args = dict(out_tokens=fake, out_num_accepted=fake, seq_offsets=fake, B=4, history=fake, capacity=16,
                lengths=fake, next_tokens=fake, device_status=None, cuda_stream=None)

    def call(**kw):
        a = dict(args); a.update(kw)
        return sv.spec_verify_commit(**a)

    assert call(B=-1) == sv.SV_ERR_INVALID_ARG
    assert call(capacity=0) == sv.SV_ERR_INVALID_ARG
    assert call(history=None) == sv.SV_ERR_INVALID_ARG
    assert call(lengths=fake + 2) == sv.SV_ERR_INVALID_ARG
    assert call(device_status=fake + 1) == sv.SV_ERR_INVALID_ARG
    assert call(B=0) == sv.SV_OK


def test_fused_host_side_checks_without_gpu(libpath):
    from speculative_decoding_verification_35_gb300 import specverify as sv
    fake = 1 << 20  # never dereferenced: every call below fails its host checks first
    args = dict(target_logits=fake, draft_logits=fake, dtype=sv.SV_BF16, draft_tokens=fake, seq_offsets=fake,
                gammas=fake, B=4, V=100, max_gamma=4, temperature=1.0, seed=1, step=0, out_tokens=fake,
                out_num_accepted=fake, device_status=None, workspace=fake, workspace_bytes=1 << 30, history=fake,
                capacity=64, lengths=fake, next_tokens=fake, cuda_stream=None)

    def call(**kw):
        a = dict(args); a.update(kw)
        return sv.spec_verify_fused(**a)

    assert call(capacity=0) == sv.SV_ERR_INVALID_ARG
    assert call(history=None) == sv.SV_ERR_INVALID_ARG
    assert call(next_tokens=fake + 2) == sv.SV_ERR_INVALID_ARG
    assert call(temperature=-1.0) == sv.SV_ERR_INVALID_ARG
    assert call(workspace=None) == sv.SV_ERR_WORKSPACE


def test_ngram_host_side_checks_without_gpu(libpath):
    from speculative_decoding_verification_35_gb300 import specverify as sv
    fake = 1 << 20  # never dereferenced: every call below returns before any CUDA call
    args = dict(history=fake, capacity=1024, lengths=fake, B=4, n_min=1, n_max=3, gamma_max=5, draft_tokens=fake,
                gammas=fake, seq_offsets=fake, match_pos=fake, device_status=None, cuda_stream=None)

    def call(**kw):
        a = dict(args); a.update(kw)
        return sv.spec_draft_ngram(**a)

    assert call(B=-1) == sv.SV_ERR_INVALID_ARG
    assert call(capacity=0) == sv.SV_ERR_INVALID_ARG
    assert call(capacity=32769) == sv.SV_ERR_INVALID_ARG
    assert call(n_min=0) == sv.SV_ERR_INVALID_ARG
    assert call(n_max=0) == sv.SV_ERR_INVALID_ARG
    assert call(gamma_max=32) == sv.SV_ERR_INVALID_ARG
    assert call(history=None) == sv.SV_ERR_INVALID_ARG
    assert call(seq_offsets=fake + 2) == sv.SV_ERR_INVALID_ARG


def test_tree_host_side_checks_without_gpu(libpath):
    from speculative_decoding_verification_35_gb300 import specverify as sv
    fake = 1 << 20  # never dereferenced: every call below fails its host checks first
    args = dict(target_logits=fake, dtype=sv.SV_BF16, draft_tokens=fake, parents=fake, seq_offsets=fake, gammas=fake,
                B=4, V=100, max_gamma=4, temperature=1.0, seed=1, step=0, out_tokens=fake, out_num_accepted=fake,
                out_path=None, device_status=None, workspace=fake, workspace_bytes=1 << 30, cuda_stream=None)

    def call(**kw):
        a = dict(args); a.update(kw)
        return sv.spec_verify_tree(**a)

    assert call(parents=None) == sv.SV_ERR_INVALID_ARG
    assert call(parents=fake + 2) == sv.SV_ERR_INVALID_ARG
    assert call(out_path=fake + 1) == sv.SV_ERR_INVALID_ARG
    assert call(max_gamma=32) == sv.SV_ERR_INVALID_ARG
    assert call(workspace=None) == sv.SV_ERR_WORKSPACE


def test_shard_host_side_checks_without_gpu(libpath):
    from speculative_decoding_verification_35_gb300 import specverify as sv
    fake = 1 << 20  # never dereferenced: every call below fails its host checks first
    st = dict(shard_target=fake, shard_draft=fake, dtype=sv.SV_BF16, draft_tokens=fake, seq_offsets=fake, gammas=fake,
              B=4, V=100, v0=50, Vs=50, max_gamma=4, temperature=1.0, partials=fake, device_status=fake,
              cuda_stream=None)

    def stats(**kw):
        a = dict(st); a.update(kw)
        return sv.spec_shard_stats(**a)

    assert stats(v0=60) == sv.SV_ERR_INVALID_ARG          # slice past V
    assert stats(Vs=0) == sv.SV_ERR_INVALID_ARG
    assert stats(partials=fake + 8) == sv.SV_ERR_INVALID_ARG  # records 16-byte aligned
    assert stats(temperature=-1.0) == sv.SV_ERR_INVALID_ARG
    assert stats(max_gamma=32) == sv.SV_ERR_INVALID_ARG
    assert stats(B=0) == sv.SV_OK
    dc = dict(all_partials=fake, S=2, bounds=[0, 50, 100], draft_tokens=fake, seq_offsets=fake, gammas=fake, B=4,
              V=100, max_gamma=4, temperature=1.0, point_mass=0, seed=1, step=0, out_tokens=fake,
              out_num_accepted=fake, draws=fake, device_status=fake, cuda_stream=None)

    def decide(**kw):
        a = dict(dc); a.update(kw)
        return sv.spec_shard_decide(**a)

    assert decide(bounds=[0, 50, 99]) == sv.SV_ERR_INVALID_ARG   # last bound must be V
    assert decide(bounds=[0, 60, 50]) == sv.SV_ERR_INVALID_ARG   # bounds increase
    assert decide(S=9, bounds=list(range(0, 99, 11)) + [100]) == sv.SV_ERR_INVALID_ARG  # at most 8 shards
    assert decide(draws=fake + 4) == sv.SV_ERR_INVALID_ARG
    assert decide(B=0) == sv.SV_OK
    assert sv.spec_shard_sums(2, 2, [0, 50, 100], fake, fake, sv.SV_BF16, fake, fake, 4, 100, 1.0, fake, None) == \
        sv.SV_ERR_INVALID_ARG  # shard index past S
    assert sv.spec_shard_sums(0, 2, [0, 50, 100], fake, fake, sv.SV_BF16, fake, fake, 4, 100, 1.0, fake + 8, None) == \
        sv.SV_ERR_INVALID_ARG  # records 16-byte aligned
    assert sv.spec_shard_sums(0, 2, [0, 50, 100], fake, fake, sv.SV_BF16, fake, fake, 4, 100, 0.0, fake, None) == \
        sv.SV_OK  # greedy: no draws
    # records per sequence: chunks of the widest shard
    assert sv.spec_shard_chunks(2, [0, 50, 100]) == 1
    assert sv.spec_shard_chunks(2, [0, 8192, 8193]) == 1
    assert sv.spec_shard_chunks(2, [0, 1, 8194]) == 2
    assert sv.spec_shard_chunks(2, [0, 64128, 128256]) == 8
    assert sv.spec_shard_chunks(4, [0, 32064, 64128, 96192, 128256]) == 4
    assert sv.spec_shard_chunks(2, [0, 60, 50]) == 0
    assert sv.spec_shard_chunks(2, [1, 60, 100]) == 0
    assert sv.spec_shard_chunks(9, list(range(0, 99, 11)) + [100]) == 0
    assert sv.spec_shard_finish(2, 2, [0, 50, 100], fake, fake, sv.SV_BF16, fake, fake, fake, 4, 100, 1.0, fake,
                                None) == sv.SV_ERR_INVALID_ARG  # shard index past S
    assert sv.spec_shard_finish(0, 2, [0, 50, 100], fake, fake, sv.SV_BF16, fake, fake, fake, 4, 100, 0.0, fake,
                                None) == sv.SV_OK  # greedy: nothing to finish


def test_host_buffer_form_checks_without_gpu(libpath):
    import numpy as np
    from speculative_decoding_verification_35_gb300 import specverify as sv
    fake = 1 << 20  # device staging addresses, never dereferenced: every call below fails its host checks
    offs = np.array([0, 4, 8, 12, 16], dtype=np.int32)  # read on the host by this entry point
    gam = np.full(4, 4, dtype=np.int32)
    dev = sv.SvDeviceBuffers(fake, fake, fake, fake, fake, fake, fake)
    args = dict(target_logits=fake, draft_logits=fake, dtype=sv.SV_BF16, draft_tokens=fake,
                seq_offsets=offs.ctypes.data, gammas=gam.ctypes.data, B=4, V=100, max_gamma=4, temperature=1.0,
                seed=1, step=0, out_tokens=fake, out_num_accepted=fake, dev=dev, device_status=None, workspace=fake,
                workspace_bytes=1 << 30, cuda_stream=None)

    def call(**kw):
        a = dict(args); a.update(kw)
        return sv.spec_verify_host(**a)

    assert call(dev=None) == sv.SV_ERR_INVALID_ARG
    assert call(max_gamma=32) == sv.SV_ERR_INVALID_ARG
    assert call(dtype=7) == sv.SV_ERR_INVALID_ARG
    assert call(seq_offsets=None) == sv.SV_ERR_INVALID_ARG
    bad = offs.copy(); bad[4] = -1
    assert call(seq_offsets=bad.ctypes.data) == sv.SV_ERR_INVALID_ARG
    bad[4] = 17  # more draft rows than B * max_gamma
    assert call(seq_offsets=bad.ctypes.data) == sv.SV_ERR_INVALID_ARG
    assert call(target_logits=None) == sv.SV_ERR_INVALID_ARG
    assert call(dev=sv.SvDeviceBuffers(fake, None, fake, fake, fake, fake, fake)) == sv.SV_ERR_INVALID_ARG
    assert call(temperature=float("nan")) == sv.SV_ERR_INVALID_ARG
    assert call(workspace=None) == sv.SV_ERR_WORKSPACE
    assert call(B=0) == sv.SV_OK


def test_binding_raises_without_the_library(tmp_path):
    """A copy of the package without its compiled library fails at import: there is no fallback path."""
    import shutil
    import sys
    src = os.path.join(ROOT, "speculative_decoding_verification_35_gb300")
    shutil.copytree(src, tmp_path / "speculative_decoding_verification_35_gb300",
                    ignore=shutil.ignore_patterns("*.so", "*.o", "csrc", "__pycache__"))
    r = subprocess.run([sys.executable, "-c", "import speculative_decoding_verification_35_gb300.specverify"],
                       cwd=tmp_path, capture_output=True, text=True, env={**os.environ, "PYTHONPATH": str(tmp_path)})
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "is not built" in r.stderr, r.stderr[-500:]
