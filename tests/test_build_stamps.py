"""The in-tree build reuses an object or the library only when the SHA-256
recorded beside it matches what it was built from (sources, every header,
flags), never by modification times: a prebuilt binary carried in with the
tree, or one whose record is missing, is rebuilt."""

import os

from kv_cache_compression_frame_gb300 import build_lib as B


def test_digest_covers_content_and_framing():
    a = B._sha(b"abc", b"def")
    assert a == B._sha(b"abc", b"def")
    assert a != B._sha(b"abcd", b"ef")          # lengths are part of the digest
    assert a != B._sha(b"abc", b"deg")


def test_stamp_needs_the_target_and_a_matching_record(tmp_path):
    obj = tmp_path / "x.o"
    assert not B._stamp_ok(str(obj), "d1")      # nothing built
    obj.write_bytes(b"\x7fELF")
    assert not B._stamp_ok(str(obj), "d1")      # a binary without its record
    B._write_stamp(str(obj), "d1")
    assert B._stamp_ok(str(obj), "d1")
    assert not B._stamp_ok(str(obj), "d2")      # sources changed since
    # a newer modification time does not make a stale record current
    os.utime(obj, (4e9, 4e9))
    assert not B._stamp_ok(str(obj), "d2")
    os.remove(str(obj))
    assert not B._stamp_ok(str(obj), "d1")      # record without the binary


def test_headers_digest_sees_every_header(tmp_path, monkeypatch):
    csrc, inc = tmp_path / "csrc", tmp_path / "include"
    csrc.mkdir()
    inc.mkdir()
    (csrc / "a.cuh").write_text("int a;")
    (inc / "b.h").write_text("int b;")
    monkeypatch.setattr(B, "CSRC", str(csrc))
    monkeypatch.setattr(B, "INCLUDE", str(inc))
    d0 = B._headers_digest()
    (inc / "b.h").write_text("int b2;")
    d1 = B._headers_digest()
    assert d1 != d0
    (csrc / "c.cuh").write_text("")
    assert B._headers_digest() != d1
