"""The library build notices an edit to any of its sources (CPU only: no
compiler run; the digest check is exercised on a copy of csrc/)."""
import shutil

import sparse_attention_mxfp4_gb300.buildlib as B


def test_every_kernel_source_is_hashed():
    names = {f.rsplit("/", 1)[-1] for f in B.source_files()}
    for want in ("mx4_index.cu", "score_kernel.cuh", "attn_kernel.cuh", "topk_kernel.cuh", "writer_kernel.cuh",
                 "sm103_ptx.cuh", "mx4_index.h"):
        assert want in names, want


def test_an_edit_to_any_source_marks_the_library_stale(tmp_path, monkeypatch):
    csrc = tmp_path / "csrc"
    shutil.copytree(B.CSRC, csrc)
    monkeypatch.setattr(B, "CSRC", str(csrc))
    lib = tmp_path / "lib.so"
    lib.write_bytes(b"not a library")
    (tmp_path / "lib.so.sha256").write_text(B.source_digest() + "\n")
    assert not B._stale(str(lib))
    sources = sorted(csrc.glob("*.cuh")) + sorted(csrc.glob("*.cu"))
    assert len(sources) >= 6
    for f in sources:
        orig = f.read_bytes()
        f.write_bytes(orig + b"\n// an edit\n")
        assert B._stale(str(lib)), f.name
        f.write_bytes(orig)
        assert not B._stale(str(lib)), f.name
    # other nvcc flags are another build
    assert B._stale(str(lib), extra_flags=("-DX=1",))
    # no recorded digest: stale
    (tmp_path / "lib.so.sha256").unlink()
    assert B._stale(str(lib))
