"""Host logic of the Python binding; no GPU is needed and nothing is launched.

* backward_path(): the backward algorithm that path="auto" (and the autograd
  function) takes for each workload's sizes. It asks the library for the
  binned workspace size, a host-only call.
* _dims(): the shape and dtype checks that turn tensors into da_dims before
  any library call.
"""
import pytest
import torch

import da_inputs
import deformable_view_feature_gb300 as da

DTYPES = {"f32": da.DA_F32, "bf16": da.DA_BF16, "f16": da.DA_F16}


@pytest.fixture(scope="module", autouse=True)
def lib():
    da.build.build()
    return da.load_library()


def _dims_of(wl):
    return da.DaDims(wl.batch, wl.num_cams, wl.num_scales, wl.num_embeds, wl.num_groups, wl.num_anchors,
                     wl.num_pts, DTYPES[wl.feat_dtype], wl.num_feat_rows)


@pytest.mark.parametrize("name,path", [
    ("sp4d_train", "binned"),   # 13*6*4 = 312 samples per (anchor, group)
    ("sp4d_inf", "binned"),
    ("large_bf16", "binned"),
    ("tiny", "scatter"),        # 4 samples per (anchor, group)
    ("dcnv4", "scatter"),       # 9
])
def test_backward_path_of_each_workload(name, path):
    assert da.backward_path(_dims_of(da_inputs.WORKLOADS[name])) == path


def test_backward_path_edges():
    base = dict(batch=2, num_cams=2, num_scales=2, num_embeds=64, num_groups=2, num_anchors=10,
                num_pts=4, feat_dtype=da.DA_F32, num_feat_rows=400)

    def path(**kw):
        d = dict(base)
        d.update(kw)
        return da.backward_path(da.DaDims(**d))

    assert path(num_pts=4) == "scatter"                        # P*K*S = 16: the small-task bound
    assert path(num_pts=5) == "binned"                         # 20
    assert path(num_pts=5, num_embeds=24, num_groups=3) == "scatter"   # C not a power of two
    assert path(num_pts=5, num_embeds=64, num_groups=16) == "scatter"  # D = 4, not a multiple of 8
    assert path(num_pts=5, num_embeds=512, num_groups=64) == "scatter"  # C above 256
    assert path(num_pts=5, num_embeds=256, num_groups=4, feat_dtype=da.DA_BF16) == "binned"
    # Record indices past int32 (4 corners per sample): the binned kernels refuse them.
    assert path(batch=1 << 20, num_anchors=1 << 10, num_pts=5) == "scatter"


def _tensors(B=1, rows=16, C=32, A=4, P=2, K=1, S=1, G=1):
    feat = torch.zeros(B, rows, C)
    ss = torch.tensor([[[4, 4]] * S] * K, dtype=torch.int32)
    loc = torch.zeros(B, A, P, K, 2)
    w = torch.zeros(B, A, P, K, S, G)
    return feat, ss, loc, w


def test_dims_from_tensors():
    feat, ss, loc, w = _tensors(B=2, rows=48, C=64, A=5, P=3, K=3, S=1, G=4)
    d = da._dims(feat, ss, loc, w)
    assert (d.batch, d.num_cams, d.num_scales, d.num_embeds, d.num_groups, d.num_anchors, d.num_pts,
            d.feat_dtype, d.num_feat_rows) == (2, 3, 1, 64, 4, 5, 3, da.DA_F32, 48)
    assert da._dims(feat.to(torch.bfloat16), ss, loc, w).feat_dtype == da.DA_BF16
    assert da._dims(feat.to(torch.float16), ss, loc, w).feat_dtype == da.DA_F16


def test_dims_reject_bad_shapes_and_types():
    feat, ss, loc, w = _tensors(K=2, S=2, G=2)
    with pytest.raises(ValueError, match="mc_ms_feat"):
        da._dims(feat[0], ss, loc, w)
    with pytest.raises(ValueError, match="sampling_location"):
        da._dims(feat, ss, loc[..., :1], w)
    with pytest.raises(ValueError, match="spatial_shape"):
        da._dims(feat, ss[:1], loc, w)
    with pytest.raises(ValueError, match="weights"):
        da._dims(feat, ss, loc, w[:, :, :, :, :1])
    with pytest.raises(ValueError, match="batch"):
        da._dims(feat, ss, torch.cat([loc, loc]), w)
    with pytest.raises(TypeError, match="mc_ms_feat"):
        da._dims(feat.double(), ss, loc, w)
    with pytest.raises(TypeError, match="float32"):
        da._dims(feat, ss, loc.double(), w)
    with pytest.raises(TypeError, match="float32"):
        da._dims(feat, ss, loc, w.half())


def test_map_tables_travel_as_host_int32():
    t = da._host_i32([[[4, 5], [2, 3]]])
    assert t.dtype == torch.int32 and t.device.type == "cpu" and t.is_contiguous()
    assert t.tolist() == [[[4, 5], [2, 3]]]
    assert da._host_i32(torch.tensor([0, 20], dtype=torch.int64)).dtype == torch.int32
