"""Checkpoint files of the long-run driver: format, hash, corruption and identity checks (host
code only, no GPU needed)."""
import struct

import numpy as np
import pytest

import qubo_instances as qi

LAYOUT = "<8sIiiiQQQiidQQ"  # everything before the trailing checksum


@pytest.fixture(scope="module")
def q():
    import exact_qubo_exhaustive_gb300 as lib
    return lib


def test_fnv1a64_published_vectors(q):
    assert q.fnv1a64(b"") == 0xCBF29CE484222325
    assert q.fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert q.fnv1a64(b"foobar") == 0x85944171F73967E8


def write_ckpt(q, path, **f):
    body = struct.pack(LAYOUT, b"QUBOCKP1", 1, f["n"], f["dtype"], f["k"], f["qh"], f["next"], f["total"],
                       f["have"], 0, f["e"], f["rank"], f["ties"])
    assert len(body) == 80
    path.write_bytes(body + struct.pack("<Q", q.fnv1a64(body)))


def test_read_back_a_written_record(q, tmp_path):
    p = tmp_path / "run.ckpt"
    write_ckpt(q, p, n=30, dtype=0, k=6, qh=123, next=16, total=64, have=1, e=-1234.0, rank=99, ties=2)
    r = q.checkpoint_read(str(p))
    assert (r["n"], r["k_prefix"], r["next_slice"], r["total_slices"]) == (30, 6, 16, 64)
    assert (r["have"], r["min_energy"], r["argmin_rank"], r["tie_count"], r["q_hash"]) == (1, -1234.0, 99, 2, 123)


def test_corrupt_truncated_and_missing_files_are_rejected(q, tmp_path):
    p = tmp_path / "run.ckpt"
    write_ckpt(q, p, n=30, dtype=0, k=6, qh=1, next=0, total=64, have=0, e=0.0, rank=0, ties=0)
    raw = bytearray(p.read_bytes())
    raw[40] ^= 1  # one flipped bit: the checksum no longer matches
    p.write_bytes(bytes(raw))
    with pytest.raises(q.QuboError) as ei:
        q.checkpoint_read(str(p))
    assert ei.value.status == -8
    p.write_bytes(bytes(raw[:50]))
    with pytest.raises(q.QuboError):
        q.checkpoint_read(str(p))
    with pytest.raises(q.QuboError):
        q.checkpoint_read(str(tmp_path / "absent.ckpt"))


def test_a_file_of_another_problem_is_refused_before_any_search(q, tmp_path):
    Q = qi.random_upper_int(20, -50, 50, 1)
    p = tmp_path / "run.ckpt"
    other = q.fnv1a64(np.ascontiguousarray(Q + 1).tobytes())
    write_ckpt(q, p, n=20, dtype=0, k=4, qh=other, next=3, total=16, have=1, e=-5.0, rank=7, ties=1)
    before = p.read_bytes()
    with pytest.raises(q.QuboError) as ei:
        q.solve_checkpointed(Q, 4, str(p))
    assert ei.value.status == -8 and p.read_bytes() == before  # left untouched


def test_argument_errors(q, tmp_path):
    Q = qi.random_upper_int(10, -5, 5, 2)
    for k in (0, 10):
        with pytest.raises(q.QuboError) as ei:
            q.solve_checkpointed(Q, k, str(tmp_path / "x.ckpt"))
        assert ei.value.status == -1
