"""The bounds-checked build against the regular one.

libnsmuon_checked.so is the library compiled with NSM_CHECKED=1: before each access to
a matrix's elements (a global load or store, a TMA box) its kernels test that the access
lies inside that matrix, record a failed test in the device status word (NSM_ERR_BOUNDS
with the kernel, role and site) and skip the access.  It stands in for a memory checker,
which this GPU pool does not offer.

The cases of tests/checked_cases.py (every kernel and access path of the library, on
odd and ragged shapes) run in a child process that loads the checked build.  No test
may fail there, and every output must equal, bit for bit, the regular build's output
on the same inputs: the checks sit beside the arithmetic and change none of it.  The
same holds for one step over each whole benchmark table (llama7b, split_moe), compared
through exact digests of the updated buffers.
"""

import json
import os
import subprocess
import sys

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def nsm():
    import newton_schulz_orthogonalized_gb300 as m
    m.lib()
    return m


@pytest.fixture(scope="module")
def checked_run(tmp_path_factory):
    import newton_schulz_orthogonalized_gb300 as m
    if not os.path.exists(m.LIB_CHECKED):
        pytest.fail(f"{m.LIB_CHECKED} is missing: __graft_entry__.build() builds it")
    path = str(tmp_path_factory.mktemp("checked") / "out.npz")
    env = dict(os.environ, NSM_CHECKED="1")
    proc = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "checked_cases.py"), path],
                          env=env, cwd=ROOT, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                          text=True, timeout=900)
    assert proc.returncode == 0, proc.stdout[-4000:]
    with open(os.path.splitext(path)[0] + ".json") as f:
        meta = json.load(f)
    data = np.load(path)
    return meta, {k: data[k] for k in data.files}


def test_bounds_selftest_regular_build_records_nothing(nsm):
    assert not nsm.checked_build()
    nsm.bounds_selftest()
    assert nsm.device_status_detail() == (nsm.NSM_OK, 0, 0, 0)


def test_bounds_selftest_checked_build_records_the_site():
    code = (
        "import newton_schulz_orthogonalized_gb300 as m\n"
        "assert m.checked_build(), m.LIB_PATH\n"
        "m.bounds_selftest()\n"
        "print(list(m.device_status_detail()))\n"
        "print(list(m.device_status_detail()))\n"
    )
    env = dict(os.environ, NSM_CHECKED="1")
    proc = subprocess.run([sys.executable, "-c", code], env=env, cwd=ROOT, stdout=subprocess.PIPE,
                          stderr=subprocess.STDOUT, text=True, timeout=300)
    assert proc.returncode == 0, proc.stdout[-4000:]
    first, second = [json.loads(line) for line in proc.stdout.strip().splitlines()[-2:]]
    import newton_schulz_orthogonalized_gb300 as m
    assert first == [m.NSM_ERR_BOUNDS, m.NSM_KERNEL_SELFTEST, 0, m.NSM_SITE_SELFTEST_BOUNDS]
    assert second == [m.NSM_OK, 0, 0, 0]  # reading the status clears it


def test_checked_build_records_no_failure(checked_run):
    meta, _ = checked_run
    assert meta["checked"] is True
    assert meta["lib"].endswith("libnsmuon_checked.so")
    failed = {name: st for name, st in meta["status"].items() if tuple(st) != (0, 0, 0, 0)}
    assert not failed, failed


def test_checked_build_matches_regular_bitwise(nsm, checked_run):
    import checked_cases
    _, checked = checked_run
    regular, status = checked_cases.run(nsm)
    assert all(tuple(st) == (0, 0, 0, 0) for st in status.values()), status
    assert sorted(regular) == sorted(checked)
    for name, want in regular.items():
        got = checked[name]
        assert got.shape == want.shape, name
        same = got.view(np.uint8) == want.view(np.uint8)
        assert same.all(), f"{name}: {int((~same).sum())} bytes differ"


@pytest.mark.slow
@pytest.mark.parametrize("name", ["llama7b", "split_moe"])
def test_checked_build_full_table_matches_regular(nsm, tmp_path, name):
    import torch

    import checked_cases
    torch.cuda.empty_cache()  # the child needs the device memory this process has cached
    path = str(tmp_path / "digest.json")
    env = dict(os.environ, NSM_CHECKED="1")
    proc = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "checked_cases.py"), "--fullsize",
                           name, path], env=env, cwd=ROOT, stdout=subprocess.PIPE,
                          stderr=subprocess.STDOUT, text=True, timeout=1200)
    assert proc.returncode == 0, proc.stdout[-4000:]
    with open(path) as f:
        checked = json.load(f)
    assert checked["checked"] is True
    assert tuple(checked["status"]) == (0, 0, 0, 0), checked["status"]
    regular = checked_cases.fullsize_digest(nsm, name)
    assert tuple(regular["status"]) == (0, 0, 0, 0)
    for key in ("params", "momentum", "copy"):
        assert checked[key] == regular[key], key
