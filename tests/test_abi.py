"""Host-side tests of the C ABI (no GPU): the library loads and exports every
symbol include/spconv.h declares, argument validation, and the packed layout
(weight stretching + output-channel binning) decodes back to the CSR input."""
import ctypes
import os
import re

import numpy as np
import pytest

import workloads
import sparse_weight_direct_gb300 as swd
from sparse_weight_direct_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "spconv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spconv_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert set(names) == set(_lib.EXPORTS)
    L = _lib.lib()
    for n in names:
        assert getattr(L, n) is not None
    # nothing else is exported
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", swd.library_path()],
                         capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert {e for e in exported if e.startswith("spconv")} == set(names)


def test_status_strings():
    for code in range(-7, 1):
        s = swd.status_string(code)
        assert s and "unknown" not in s
    assert "unknown" in swd.status_string(-99)


def _pack_host(L, rowptr, colidx, value, fmt="f32"):
    return swd.pack_host(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=L.R, S=L.S,
                         stride=L.stride, pad=L.pad, fmt=fmt)


def decode_layout(w):
    """Rebuild {m: sorted [(colidx, value)]} from the packed blobs."""
    info = w.info()
    blobs = w.array("blobs")
    boff = w.array("blob_off").astype(np.int64) * 16
    head_oc = w.array("slot_oc")
    nxt = w.array("slot_next")
    flags = w.array("group_flags")
    st, R, S = info["stride"], info["R"], info["S"]
    G, nch, hw = info["groups"], info["num_chunks"], info["hdr_words"]
    spg = info["warps"] * info["slots_per_warp"]
    assert flags.size == G and head_oc.size == nxt.size == G * spg
    # owner of every slot: follow each head's chain of parts
    slot_oc = np.full(G * spg, -1, dtype=np.int64)
    for g in range(G):
        for ls in range(spg):
            m = int(head_oc[g * spg + ls])
            if m < 0:
                continue
            c, seen = ls, 0
            while c >= 0:
                assert slot_oc[g * spg + c] == -1  # a slot belongs to one chain
                slot_oc[g * spg + c] = m
                c = int(nxt[g * spg + c])
                seen += 1
            if seen > 1:
                assert flags[g] & 2
        assert bool(flags[g] & 1) == (g < info["dense_groups"])
    assert boff.size == G * nch + 1 and boff[-1] == blobs.size
    assert np.all(boff % 16 == 0) and np.all(np.diff(boff) >= hw * 4)
    rows = {}
    RS = R * info["S"]
    kk4 = (RS + 3) // 4 * 4
    Q, NW, chunk = info["slots_per_warp"], info["warps"], info["chunk"]
    for g in range(G):
        for k in range(nch):
            blob = blobs[boff[g * nch + k]:boff[g * nch + k + 1]]
            assert blob.size <= info["blob_stage_bytes"]
            if g < info["dense_groups"]:
                mw = info["dense_mask_words"]
                mask = blob[:mw * 4].view(np.uint32)[:NW * chunk].reshape(NW, chunk)
                wts = blob[mw * 4:].view(np.float32).reshape(NW, chunk, Q, kk4)
                assert np.all(wts[..., RS:] == 0)
                for w in range(NW):
                    for q in range(Q):
                        m = int(slot_oc[(g * NW + w) * Q + q])
                        for cl in range(chunk):
                            blk = wts[w, cl, q, :RS]
                            present = bool(mask[w, cl] >> q & 1)
                            if m < 0 or not present:
                                assert not blk.any()
                                continue
                            c = k * chunk + cl
                            assert c < info["C"]
                            for t in np.nonzero(blk)[0]:
                                rows.setdefault(m, []).append((c * RS + int(t), float(blk[t])))
                continue
            hdr = blob[:hw * 4].view(np.uint32)
            assert hdr[0] == 0 and np.all(np.diff(hdr[:spg + 1].astype(np.int64)) >= 0)
            if info["format"] == 1:
                # [31:16] fp16 value, [15:8] channel in chunk, [7:4] column, [3:0] row
                words = blob[hw * 4:].view(np.uint32)
                assert hdr[spg] <= words.size
                # padding past the last word: to 16 bytes, or to the fixed blob stride
                assert info["blob_stride"] or words.size - hdr[spg] <= 3
                assert not words[hdr[spg]:].any()
                for ls in range(spg):
                    m = int(slot_oc[g * spg + ls])
                    seg = words[hdr[ls]:hdr[ls + 1]]
                    if m < 0:
                        assert seg.size == 0
                        continue
                    for wd in seg.tolist():
                        v = float(np.array([wd >> 16], np.uint16).view(np.float16)[0])
                        cl, s, r = (wd >> 8) & 0xFF, (wd >> 4) & 0xF, wd & 0xF
                        assert cl < info["chunk"] and r < R and s < S
                        c = k * info["chunk"] + cl
                        rows.setdefault(m, []).append(((c * R + r) * S + s, v))
                continue
            ent = blob[hw * 4:].view([("value", "<f4"), ("off", "<i4")])
            end = int(hdr[spg])
            if info["tap_pairs"]:
                # pair ranges after the single ranges; 16-byte pair entries
                NP = Q * (Q - 1) // 2
                assert Q in (2, 4) and hw == (spg + 1 + NW * NP + 1 + 3) // 4 * 4
                hp = hdr[spg + 1:spg + 2 + NW * NP].astype(np.int64)
                assert hp[0] == (end + 1) // 2 * 2 and np.all(np.diff(hp) >= 0)
                assert np.all(hp % 2 == 0)
                pair_of = [(a, b) for a in range(Q) for b in range(a + 1, Q)]
                for w in range(NW):
                    for pi, (q1, q2) in enumerate(pair_of):
                        seg = blob[hw * 4 + 8 * hp[w * NP + pi]:hw * 4 + 8 * hp[w * NP + pi + 1]]
                        pe = seg.view([("va", "<f4"), ("vb", "<f4"), ("off", "<i4"), ("z", "<i4")])
                        assert not pe["z"].any()
                        for q, key in ((q1, "va"), (q2, "vb")):
                            m = int(slot_oc[(g * NW + w) * Q + q])
                            assert m >= 0 or pe.size == 0
                            for e in pe:
                                off = int(e["off"])
                                cl, rem = divmod(off - (info["shift"] if st == 1 else 0),
                                                 info["plane"])
                                r, qq = divmod(rem, info["row_pitch"])
                                if st == 1:
                                    s = qq
                                else:
                                    phase, qq2 = divmod(qq, info["phase_pitch"])
                                    s = qq2 * st + phase
                                c = k * info["chunk"] + cl
                                rows.setdefault(m, []).append(((c * R + r) * S + s, float(e[key])))
                end = int(hp[-1])
            assert end <= ent.size
            # padding past the last entry: to 16 bytes (with pairs, plus the 8 bytes
            # reserved for their alignment), or to the fixed blob stride
            assert info["blob_stride"] or ent.size - end <= (3 if info["tap_pairs"] else 1)
            assert not blob[hw * 4 + 8 * end:].any()
            for ls in range(spg):
                m = int(slot_oc[g * spg + ls])
                seg = ent[hdr[ls]:hdr[ls + 1]]
                if m < 0:
                    assert seg.size == 0
                    continue
                for e in seg:
                    off = int(e["off"])
                    if info["plane_stage"]:
                        # raw planes after 16 zeroed words; low bits flag the
                        # sides the tap can leave the image by
                        flags, off = off & 15, (off >> 4) - 16 + info["W"] + 1
                        cl, rem = divmod(off, info["plane"])
                        r, s = divmod(rem, info["W"])
                        assert flags == (s == 0) | (s == 2) << 1 | (r == 0) << 2 | (r == 2) << 3
                    elif st == 1:
                        # (the shift is -1 on tight-pitch plans: decode from the
                        # tap's distance to the channel's first staged word)
                        cl, rem = divmod(off - info["shift"], info["plane"])
                        r, s = divmod(rem, info["row_pitch"])
                    else:
                        cl, rem = divmod(off, info["plane"])
                        r, q = divmod(rem, info["row_pitch"])
                        phase, qq = divmod(q, info["phase_pitch"])
                        assert phase < st
                        s = qq * st + phase
                    assert 0 <= cl < info["chunk"] and r < R and 0 <= s < S
                    c = k * info["chunk"] + cl
                    assert c < info["C"]
                    rows.setdefault(m, []).append(((c * R + r) * S + s, float(e["value"])))
    for m in rows:
        rows[m].sort()
    return info, rows, slot_oc


@pytest.mark.parametrize("fmt,name", [(f, n) for f in ("f32", "packed32") for n in (
    "tiny", "tiny_int", "resnet3x3", "vgg3x3", "sweep50", "sweep80", "sweep90", "sweep99",
    "alex11x11", "conv5x5")])
def test_packed_layout_decodes_to_csr(name, fmt):
    L = workloads.LAYERS[name]
    rowptr, colidx, value = workloads.make_weights(L)
    if fmt == "packed32":  # the format stores FP16 values (round to nearest even)
        value = value.astype(np.float16).astype(np.float32)
    w = _pack_host(L, rowptr, colidx, value, fmt)
    info, rows, slot_oc = decode_layout(w)
    assert info["on_device"] == 0 and info["nnz"] == colidx.size == info["entries"]
    assert info["in_stage_bytes"] + info["blob_stage_bytes"] <= 110 * 1024
    assert info["E"] == L.E and info["F"] == L.F
    assert info["num_slots"] == info["groups"] * info["warps"] * info["slots_per_warp"]
    # every output channel heads exactly one chain of slots
    heads = w.array("slot_oc")
    assert sorted(heads[heads >= 0].tolist()) == list(range(L.M))
    for m in range(L.M):
        lo, hi = rowptr[m], rowptr[m + 1]
        want = sorted((c, v) for c, v in zip(colidx[lo:hi].tolist(),
                                              value[lo:hi].astype(np.float64).tolist()) if v != 0)
        got = [(c, v) for c, v in rows.get(m, []) if v != 0]
        assert got == want
    # staged input tile covers every tap of every output of a tile
    if info["col_blocks"]:
        # lane_rows rows of 32 / lane_rows lanes, each lane tile_rows
        # consecutive outputs of its row; the lanes' first inputs
        # (ly * row_pitch + lx * tile_rows) fall in 32 distinct banks
        P, LR = info["tile_rows"], info["lane_rows"]
        tile_h = LR
        if info["tile_images"] == 2:
            # image pairs: lanes 0..3 of a row on the first image's sub-tile,
            # lanes 4..7 on the second's, pair_off words later
            assert LR == 4 and info["tile_cols"] == 4 * P and L.stride == 1
            assert info["pair_off"] % 32 == 16
            assert info["pair_off"] >= info["chunk"] * info["plane"]
            assert info["in_stage_bytes"] >= 4 * (info["pair_off"] + info["chunk"] * info["plane"])
            banks = {((lx // 4) * info["pair_off"] + ly * info["row_pitch"] + (lx % 4) * P) % 32
                     for ly in range(LR) for lx in range(8)}
        else:
            assert info["tile_images"] == 1 and info["pair_off"] == 0
            assert info["tile_cols"] == (32 // LR) * P and L.stride == 1
            banks = {(ly * info["row_pitch"] + lx * P) % 32 for ly in range(LR)
                     for lx in range(32 // LR)}
        assert len(banks) == 32
        assert info["row_pitch"] % 4 == 0 and info["row_pitch"] >= info["shift"] + info["in_cols"]
    else:
        tile_h = info["tile_rows"] * info["lane_rows"]
        assert info["tile_cols"] * info["lane_rows"] == 32
    if info["plane_stage"]:  # whole raw planes, the padding applied to the weights
        assert info["in_rows"] == L.H == tile_h and info["in_cols"] == L.W <= info["tile_cols"]
    elif info["shift"] == -1:  # tight pitch: 32 columns from column 0, the halo implicit
        assert info["in_rows"] == (tile_h - 1) * L.stride + L.R
        assert info["in_cols"] == info["row_pitch"] == 32 and L.W <= 31 and info["tiles_x"] == 1
    else:
        assert info["in_rows"] == (tile_h - 1) * L.stride + L.R
        assert info["in_cols"] == (info["tile_cols"] - 1) * L.stride + L.S
    assert info["tiles_y"] * tile_h >= L.E
    assert info["tiles_x"] * info["tile_cols"] >= L.F
    assert info["smem_bytes"] <= 200 * 1024
    w.close()


@pytest.mark.parametrize("hint", [0, 1, "batch"])
@pytest.mark.parametrize("name", ["tiny", "resnet3x3", "vgg3x3", "sweep50", "sweep90",
                                  "sweep99", "conv5x5"])
def test_fixed_stride_blobs(name, hint):
    """Blobs of nearly equal size (padding each to the largest adds at most a
    quarter) sit at a fixed stride, so a block finds its blob from its
    (group, chunk) index alone; otherwise they are packed back to back."""
    L = workloads.LAYERS[name]
    rowptr, colidx, value = workloads.make_weights(L)
    w = swd.pack_host(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=L.R, S=L.S,
                      stride=L.stride, pad=L.pad, batch_hint=L.N if hint == "batch" else hint)
    info = w.info()
    off = w.array("blob_off").astype(np.int64)
    sizes = np.diff(off) * 16
    stride = info["blob_stride"]
    if stride:
        assert np.all(sizes == stride) and stride % 16 == 0
        assert stride <= info["blob_stage_bytes"]
    else:
        assert sizes.max() * sizes.size > 1.25 * sizes.sum()
    if hint == "batch" and name in ("tiny", "resnet3x3", "vgg3x3"):
        assert stride > 0  # the benchmark's plans of the Bernoulli layers: near-equal blobs
    w.close()


def test_launch_plans():
    """The launch a forward would make (host logic): one-image layers split
    their channel chunks over a cluster and reduce by pushing partial sums;
    batched layers fill the GPU without a cluster; the weight-stationary
    format launches one block per (output channel, tile, image)."""
    def plan(name, N, **kw):
        L = workloads.LAYERS[name]
        rowptr, colidx, value = workloads.make_weights(L)
        w = swd.pack_host(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=L.R, S=L.S,
                          stride=L.stride, pad=L.pad, **kw)
        info, launch = w.info(), w.launch_info(N)
        w.close()
        return L, info, launch

    L, info, pl = plan("resnet3x3", 1, batch_hint=1)
    # 56-byte rows: no TMA; raw planes by one bulk copy, one block per SM
    assert info["plane_stage"] == 1 and info["chunk"] == 64
    assert pl["kernel"] == 0 and pl["cluster"] == 4 and pl["push"] == 1
    assert pl["pdl"] == 1  # one wave: start-up overlaps the previous kernel
    assert pl["grid_x"] * pl["grid_y"] == 4 * info["groups"] <= 152 and pl["grid_z"] == 1
    assert pl["block_threads"] == 256 and pl["tma"] == 0
    assert pl["smem_bytes"] <= 200 * 1024
    assert info["col_blocks"] == 0
    L, info, pl = plan("vgg3x3", 16, batch_hint=16)
    assert pl["cluster"] == 1 and pl["push"] == 0 and pl["tma"] == 1 and pl["pdl"] == 1
    assert pl["grid_x"] * pl["grid_y"] == 16 * info["tiles_y"] * info["tiles_x"] * info["groups"]
    # 56 wide: column blocks, 8 x 28 tiles (two per row band), no idle lane
    assert info["col_blocks"] == 1 and info["plane_stage"] == 0
    assert (info["lane_rows"], info["tile_rows"], info["tile_cols"]) == (8, 7, 28)
    assert (info["tiles_y"], info["tiles_x"], info["row_pitch"]) == (7, 2, 36)
    L, info, pl = plan("vgg3x3", 16, batch_hint=16, fmt="packed32")
    assert info["col_blocks"] == 1  # the 32-bit words decode to the same offsets
    L, info, pl = plan("resnet3x3", 1, batch_hint=1, fmt="packed32")
    assert info["plane_stage"] == 0 and info["col_blocks"] == 0  # padded tile
    # 28 wide, dense-tap rows holding most nonzeros: image-pair column blocks
    L, info, pl = plan("sweep50", 8, batch_hint=8)
    assert info["col_blocks"] == 1 and info["tile_images"] == 2 and info["lane_rows"] == 4
    assert (info["tile_rows"], info["tile_cols"], info["tiles_y"], info["tiles_x"]) == (7, 28, 7, 1)
    # 4 image pairs x 7 row bands; most groups dense-tap: every tile's chunks split over a
    # two-block cluster, halving the long dense-tap blocks
    assert pl["grid_x"] * pl["grid_y"] == 4 * 7 * info["groups"] * 2 and pl["cluster"] == 2
    assert 2 * info["dense_groups"] >= info["groups"]
    assert info["dense_groups"] > 0
    L, info, pl = plan("sweep90", 8, batch_hint=8)  # mostly sparse rows: column-per-lane tiles
    assert info["col_blocks"] == 0 and info["lane_rows"] == 1 and info["tile_cols"] == 32
    L, info, pl = plan("sweep50", 1, batch_hint=1)  # one image: no image pairs
    assert info["tile_images"] == 1
    L, info, pl = plan("sweep80", 8, batch_hint=8)  # dense-tap groups, several waves
    assert info["dense_groups"] > 0 and pl["grid_x"] * pl["grid_y"] > 2 * 152
    assert pl["pdl"] == 0
    L, info, pl = plan("vgg3x3", 16, fmt="ws")
    assert pl["kernel"] == 1 and pl["cluster"] == 1
    assert (pl["grid_x"], pl["grid_y"], pl["grid_z"]) == (L.M, info["tiles_y"] * info["tiles_x"],
                                                          16)
    # split rows keep a cluster on the reduction by remote reads
    rng = np.random.default_rng(3)
    C, M, CRS = 128, 64, 128 * 9
    rows = [np.nonzero(rng.random(CRS) < (0.9 if m in (0, 40) else 0.1))[0] for m in range(M)]
    rowptr = np.concatenate([[0], np.cumsum([r.size for r in rows])]).astype(np.int32)
    colidx = np.concatenate(rows).astype(np.int32)
    value = np.ones(colidx.size, np.float32)
    w = swd.pack_host(rowptr, colidx, value, C=C, H=14, W=14, M=M, R=3, S=3, stride=1, pad=1,
                      batch_hint=1)
    assert (w.array("group_flags") & 2).any()
    pl = w.launch_info(1)
    assert pl["cluster"] > 1 and pl["push"] == 0
    with pytest.raises(swd.SpconvError):
        w.launch_info(0)
    w.close()


@pytest.mark.parametrize("name", ["sweep90", "sweep95", "sweep99", "vgg3x3"])
def test_binning_balances_warps(name):
    # split rows + longest-first binning keep the heaviest warp of the sparse
    # groups close to the mean (lognormal rows reach ~10x the mean row)
    L = workloads.LAYERS[name]
    rowptr, colidx, value = workloads.make_weights(L)
    w = _pack_host(L, rowptr, colidx, value)
    info = w.info()
    # (eight slots per warp on sweep99 leave coarser room: 1.6x)
    assert info["max_warp_nnz"] <= 1.6 * info["mean_warp_nnz"] + 8
    w.close()


def test_unsorted_columns_pack_like_sorted():
    rng = np.random.default_rng(0)
    M, C, R = 12, 5, 3
    rowptr, colidx, value = workloads.random_csr(M, C * R * R, 0.3, rng)
    perm_cols = colidx.copy()
    perm_vals = value.copy()
    for m in range(M):
        lo, hi = rowptr[m], rowptr[m + 1]
        p = rng.permutation(hi - lo)
        perm_cols[lo:hi] = colidx[lo:hi][p]
        perm_vals[lo:hi] = value[lo:hi][p]
    kw = dict(C=C, H=9, W=9, M=M, R=R, S=R, stride=1, pad=1)
    a = swd.pack_host(rowptr, colidx, value, **kw)
    b = swd.pack_host(rowptr, perm_cols, perm_vals, **kw)
    for k in ("blobs", "blob_off", "slot_oc", "slot_next", "group_flags"):
        np.testing.assert_array_equal(a.array(k), b.array(k))


def _status_of(**kw):
    base = dict(rowptr=np.array([0, 1], np.int32), colidx=np.array([0], np.int32),
                value=np.array([1.0], np.float32), C=1, H=5, W=5, M=1, R=3, S=3, stride=1,
                pad=1)
    base.update(kw)
    try:
        swd.pack_host(base.pop("rowptr"), base.pop("colidx"), base.pop("value"), **base).close()
        return 0
    except swd.SpconvError as e:
        return e.status


def test_packed32_limits():
    rowptr = np.array([0, 1], np.int32)
    colidx, value = np.array([0], np.int32), np.array([1.0], np.float32)
    with pytest.raises(swd.SpconvError) as e:
        swd.pack_host(rowptr, colidx, value, C=1, H=40, W=40, M=1, R=17, S=3, stride=1, pad=1,
                      fmt="packed32")
    assert e.value.status == _lib.SPCONV_ERR_UNSUPPORTED
    h = ctypes.c_void_p()
    rc = _lib.lib().spconv_pack_ex(1, 5, 5, 1, 3, 3, 1, 1, rowptr.ctypes.data_as(ctypes.c_void_p),
                                   colidx.ctypes.data_as(ctypes.c_void_p),
                                   value.ctypes.data_as(ctypes.c_void_p), 9, 0, 1, None,
                                   ctypes.byref(h))
    assert rc == _lib.SPCONV_ERR_INVALID_ARG


def test_pack_validation():
    assert _status_of() == 0
    assert _status_of(rowptr=np.array([1, 1], np.int32)) == _lib.SPCONV_ERR_BAD_CSR
    assert _status_of(rowptr=np.array([0, 2, 1], np.int32), M=2) == _lib.SPCONV_ERR_BAD_CSR
    assert _status_of(colidx=np.array([9], np.int32)) == _lib.SPCONV_ERR_BAD_CSR
    assert _status_of(colidx=np.array([-1], np.int32)) == _lib.SPCONV_ERR_BAD_CSR
    assert _status_of(rowptr=np.array([0, 2], np.int32), colidx=np.array([4, 4], np.int32),
                      value=np.array([1, 2], np.float32)) == _lib.SPCONV_ERR_BAD_CSR
    assert _status_of(C=0) == _lib.SPCONV_ERR_INVALID_ARG
    assert _status_of(stride=0) == _lib.SPCONV_ERR_INVALID_ARG
    assert _status_of(pad=-1) == _lib.SPCONV_ERR_INVALID_ARG
    assert _status_of(H=1, pad=0) == _lib.SPCONV_ERR_INVALID_ARG  # E < 1
    assert _status_of(stride=1000) == _lib.SPCONV_ERR_UNSUPPORTED
    # explicit zero weights and empty rows are fine
    assert _status_of(value=np.array([0.0], np.float32)) == 0
    assert _status_of(rowptr=np.array([0, 0], np.int32), colidx=np.zeros(0, np.int32),
                      value=np.zeros(0, np.float32)) == 0


def test_forward_rejects_host_only_handle_and_null():
    L = _lib.lib()
    rowptr = np.array([0, 1], np.int32)
    w = swd.pack_host(rowptr, np.array([4], np.int32), np.array([1.0], np.float32),
                      C=1, H=5, W=5, M=1, R=3, S=3, stride=1, pad=1)
    rc = L.spconv_forward(1, 1, 5, 5, 1, 3, 3, 1, 1, None, w.handle, None, None)
    assert rc == _lib.SPCONV_ERR_MISMATCH
    rc = L.spconv_forward(1, 1, 5, 5, 2, 3, 3, 1, 1, None, w.handle, None, None)
    assert rc == _lib.SPCONV_ERR_MISMATCH
    rc = L.spconv_forward(1, 1, 5, 5, 1, 3, 3, 1, 1, None, None, None, None)
    assert rc == _lib.SPCONV_ERR_INVALID_ARG
    L.spconv_packed_free(None)
    info = _lib.PackedInfo()
    assert L.spconv_packed_info_get(None, ctypes.byref(info)) == _lib.SPCONV_ERR_INVALID_ARG
    w.close()


def test_launch_smem_within_limit_for_any_batch():
    """Whatever batch size a plan was made for, a forward of any batch size asks
    for at most the kernels' 200 KB of dynamic shared memory (the stages a block
    runs depend on the chunks it gets, which depend on the launch's batch and
    its cluster split)."""
    for name, L in workloads.ALL_LAYERS.items():
        rowptr, colidx, value = workloads.make_weights(L)
        for hint in (0, 1, 4, 32, L.N):
            w = swd.pack_host(rowptr, colidx, value, C=L.C, H=L.H, W=L.W, M=L.M, R=L.R,
                              S=L.S, stride=L.stride, pad=L.pad, batch_hint=hint)
            for n in (1, 2, 4, 16, 64, L.N):
                li = w.launch_info(n)
                assert li["smem_bytes"] <= 200 * 1024, (name, hint, n, li["smem_bytes"])
            w.close()


SHAPE_CASES = [
    # (N hint, C, H, W, M, pad, density, plan): ad-hoc 3x3 stride-1 shapes and the
    # plan they take -- column blocks (56 / 84 / 112 wide), plane staging (14 wide
    # or less, rows TMA cannot address) or the column-per-lane padded tile
    (2, 20, 56, 56, 40, 1, 0.1, "cols"),
    (3, 9, 44, 84, 17, 1, 0.2, "cols"),     # 44 rows: the last 8-row tile half used
    (1, 6, 58, 58, 12, 0, 0.3, "cols"),
    (1, 7, 54, 54, 10, 2, 0.3, "cols"),
    (2, 12, 112, 112, 16, 1, 0.05, "cols"),
    (1, 40, 14, 10, 24, 1, 0.3, "plane"),
    (1, 64, 14, 14, 70, 1, 0.2, "plane"),
    (2, 17, 28, 28, 33, 1, 0.15, "tile"),   # 28 x 28, sparse rows: column-per-lane tiles
    (2, 17, 28, 28, 33, 1, 0.4, "cols"),    # dense rows: image-pair column blocks
    (1, 17, 28, 28, 33, 1, 0.4, "tile"),    # one image: column-per-lane tiles
    (4, 5, 30, 25, 9, 0, 0.4, "cols"),      # 28 x 23 outputs, pad 0: image pairs
    (4, 6, 20, 26, 11, 1, 0.45, "cols"),    # 20 x 26: the last 4 x 28 columns partly used
]


@pytest.mark.parametrize("case", SHAPE_CASES, ids=[str(c) for c in SHAPE_CASES])
@pytest.mark.parametrize("fmt", ["f32", "packed32"])
def test_layout_decodes_for_ad_hoc_shapes(case, fmt):
    """Whatever plan a shape takes (column blocks, plane staging, the plain
    padded tile), every packed entry decodes back to its CSR nonzero and the
    staged tile covers the output."""
    N, C, H, W, M, pad, d, plan = case
    rng = np.random.default_rng(sum(case[1:5]))
    rowptr, colidx, value = workloads.random_csr(M, C * 9, d, rng)
    if fmt == "packed32":
        value = value.astype(np.float16).astype(np.float32)
    w = swd.pack_host(rowptr, colidx, value, C=C, H=H, W=W, M=M, R=3, S=3, stride=1, pad=pad,
                      fmt=fmt, batch_hint=N)
    info, rows, _ = decode_layout(w)
    for m in range(M):
        lo, hi = rowptr[m], rowptr[m + 1]
        want = sorted((c, v) for c, v in zip(colidx[lo:hi].tolist(),
                                              value[lo:hi].astype(np.float64).tolist()) if v != 0)
        assert [(c, v) for c, v in rows.get(m, []) if v != 0] == want
    E, F = H + 2 * pad - 2, W + 2 * pad - 2
    tile_h = info["lane_rows"] if info["col_blocks"] else info["tile_rows"] * info["lane_rows"]
    assert info["tiles_y"] * tile_h >= E and info["tiles_x"] * info["tile_cols"] >= F
    got = "cols" if info["col_blocks"] else "plane" if info["plane_stage"] else "tile"
    # the 32-bit word format takes column blocks but not plane staging
    assert got == ("tile" if plan == "plane" and fmt == "packed32" else plan)
    assert info["smem_bytes"] <= 200 * 1024
    w.close()
