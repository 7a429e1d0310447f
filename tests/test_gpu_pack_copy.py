"""GPU parity of fields_copy and weno_pack_copy (the conservative-variable
copy, alone and fused with the WENO input pack) against the CPU oracle,
through the C ABI.  Both are bit copies and must match bit for bit, NaN
payloads and signed zeros included; every output array carries a canary tail
that must stay untouched."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from finite_volume_field_gb300 import api, inputs
from tests.gpu_util import assert_bits_equal, canary_intact, guarded, to_host, torch_cuda

pytestmark = pytest.mark.gpu

SMALL = [((3, 4, 5), 1), ((3, 4, 5), 2), ((5, 4, 1), 2), ((6, 3, 2), 3), ((2, 7, 3), 0),
         ((33, 31, 35), 3), ((70, 3, 40), 2), ((1, 1, 1), 2), ((40, 1, 1), 1), ((1, 37, 1), 2),
         ((65, 66, 1), 2), ((29, 34, 3), 3)]


def _dev_fields(torch, fields, offset=0):
    """Device copies of the fields; with ``offset`` 1 each starts one element
    into its allocation (8-byte but not 16-byte aligned)."""
    out = []
    for f in fields:
        whole = torch.empty(f.size + offset, dtype=torch.float64, device="cuda")
        view = whole[offset:]
        view.copy_(torch.from_numpy(np.ascontiguousarray(f)))
        out.append(view)
    return out


def _copy_outputs(torch, nv, n, offset=0):
    wholes, views = [], []
    for _ in range(nv):
        whole, view = guarded(torch, n + offset, torch.float64)
        wholes.append(whole)
        views.append(view[offset:])
    return wholes, views


def _check_copies(torch, wholes, views, fields, n, offset, what):
    torch.cuda.synchronize()
    for i, (w, v, f) in enumerate(zip(wholes, views, fields)):
        assert canary_intact(torch, w, n + offset), f"{what}: copy {i} wrote past its end"
        assert_bits_equal(to_host(v), f, what=f"{what} copy {i}")


@pytest.mark.parametrize("extents,g", SMALL)
@pytest.mark.parametrize("direction", [0, 1, 2])
@pytest.mark.parametrize("nv", [1, 3, 9])
def test_pack_copy_small(extents, g, direction, nv):
    torch = torch_cuda()
    fields = inputs.normal_fields(inputs.config_seed(3), nv, extents, g)
    n = fields[0].size
    M = oracle.pack_extents(extents, g, direction)
    npk = M[0] * M[1] * M[2] * nv
    whole_out, out = guarded(torch, npk, torch.float64)
    wholes, views = _copy_outputs(torch, nv, n)
    api.weno_pack_copy(_dev_fields(torch, fields), nv, extents, g, direction, out, views)
    torch.cuda.synchronize()
    assert canary_intact(torch, whole_out, npk), "pack wrote past its output"
    want_pack, want_copies = oracle.weno_pack_copy(fields, extents, g, direction)
    what = f"pack_copy {extents} g={g} dir={direction} nv={nv}"
    assert_bits_equal(to_host(out), want_pack, what=what)
    _check_copies(torch, wholes, views, want_copies, n, 0, what)


@pytest.mark.parametrize("extents,g", [((3, 4, 5), 1), ((33, 31, 35), 3), ((1, 1, 1), 2),
                                       ((64, 64, 1), 2), ((7, 1, 1), 0)])
@pytest.mark.parametrize("nv", [1, 2, 9])
@pytest.mark.parametrize("offset", [0, 1])
def test_fields_copy_small(extents, g, nv, offset):
    """Even and odd stored sizes; 16-byte aligned pointers (the paired-element
    path) and pointers one element in (the single-element path)."""
    torch = torch_cuda()
    fields = inputs.normal_fields(inputs.config_seed(5), nv, extents, g)
    n = fields[0].size
    wholes, views = _copy_outputs(torch, nv, n, offset)
    api.fields_copy(_dev_fields(torch, fields, offset), nv, extents, g, views)
    _check_copies(torch, wholes, views, oracle.fields_copy(fields, extents, g), n, offset,
                  f"copy {extents} g={g} nv={nv} offset={offset}")


def test_pack_copy_special_bits_and_max_nv():
    """NaN payloads, -0.0, infinities and subnormals copy bit for bit through
    both outputs; 64 variables (the maximum) all land in place."""
    torch = torch_cuda()
    extents, g = (9, 10, 11), 2
    n = int(np.prod(inputs.stored_extents(extents, g)))
    fields = []
    for i in range(64):
        b = inputs.random_bits(19, i, n)
        b[::7] = 0x7FF4DEADBEEF0000 + i
        b[1::11] = 0x8000000000000000
        b[2::13] = 0x0000000000000003
        b[3::17] = 0xFFF0000000000000
        fields.append(b.view(np.float64))
    dev = _dev_fields(torch, fields)
    for direction in range(3):
        M = oracle.pack_extents(extents, g, direction)
        npk = M[0] * M[1] * M[2] * 64
        whole_out, out = guarded(torch, npk, torch.float64)
        wholes, views = _copy_outputs(torch, 64, n)
        api.weno_pack_copy(dev, 64, extents, g, direction, out, views)
        torch.cuda.synchronize()
        assert canary_intact(torch, whole_out, npk)
        want_pack, want_copies = oracle.weno_pack_copy(fields, extents, g, direction)
        assert_bits_equal(to_host(out), want_pack, what=f"dir {direction}")
        _check_copies(torch, wholes, views, want_copies, n, 0, f"dir {direction}")
    wholes, views = _copy_outputs(torch, 64, n)
    api.fields_copy(dev, 64, extents, g, views)
    _check_copies(torch, wholes, views, fields, n, 0, "fields_copy 64")


def test_copy_aliasing_rules():
    """Fields may repeat; a copy overlapping a field, another copy or the
    packed output is refused with nothing launched."""
    torch = torch_cuda()
    extents, g = (8, 9, 10), 1
    f = inputs.normal_fields(7, 1, extents, g)[0]
    n = f.size
    dev = _dev_fields(torch, [f])[0]
    M = oracle.pack_extents(extents, g, 1)
    out = torch.empty(M[0] * M[1] * M[2] * 3, dtype=torch.float64, device="cuda")
    copies = [torch.empty(n, dtype=torch.float64, device="cuda") for _ in range(3)]
    api.weno_pack_copy([dev, dev, dev], 3, extents, g, 1, out, copies)
    torch.cuda.synchronize()
    want_pack, _ = oracle.weno_pack_copy([f, f, f], extents, g, 1)
    assert_bits_equal(to_host(out), want_pack)
    for c in copies:
        assert_bits_equal(to_host(c), f)
    big = torch.zeros(4 * n, dtype=torch.float64, device="cuda")
    before = api.launch_count()
    cases = [
        lambda: api.fields_copy([dev], 1, extents, g, [dev]),
        lambda: api.fields_copy([dev, dev], 2, extents, g, [big[:n], big[n // 2: n // 2 + n]]),
        lambda: api.weno_pack_copy([dev], 1, extents, g, 0, big[:n], [big[n // 2: n // 2 + n]]),
        lambda: api.weno_pack_copy([dev], 1, extents, g, 2, big[:n], [dev]),
    ]
    for case in cases:
        with pytest.raises(api.FvfError) as e:
            case()
        assert e.value.status == 6
    assert api.launch_count() == before
    torch.cuda.synchronize()


def test_pack_copy_full_size_207_cubed():
    """8 fields of 201^3 interior + 3 ghost layers (207^3 stored), N(0,1):
    the fused pack and copy along x, y and z, and the copy alone, every
    element compared with the oracle."""
    torch = torch_cuda()
    extents, g, nv = (201, 201, 201), 3, 8
    fields = inputs.normal_fields(inputs.config_seed(3), nv, extents, g)
    dev = _dev_fields(torch, fields)
    n = fields[0].size
    M = oracle.pack_extents(extents, g, 0)
    out = torch.empty(M[0] * M[1] * M[2] * nv, dtype=torch.float64, device="cuda")
    copies = [torch.empty(n, dtype=torch.float64, device="cuda") for _ in range(nv)]
    for direction in range(3):
        out.fill_(0.0)
        for c in copies:
            c.fill_(0.0)
        api.weno_pack_copy(dev, nv, extents, g, direction, out, copies)
        torch.cuda.synchronize()
        want_pack, want_copies = oracle.weno_pack_copy(fields, extents, g, direction)
        assert_bits_equal(to_host(out), want_pack, what=f"207^3 dir {direction}")
        for i, c in enumerate(copies):
            assert_bits_equal(to_host(c), want_copies[i], what=f"207^3 dir {direction} copy {i}")
    for c in copies:
        c.fill_(0.0)
    api.fields_copy(dev, nv, extents, g, copies)
    torch.cuda.synchronize()
    want_copies = oracle.fields_copy(fields, extents, g)
    for i, c in enumerate(copies):
        assert_bits_equal(to_host(c), want_copies[i], what=f"207^3 fields_copy {i}")
