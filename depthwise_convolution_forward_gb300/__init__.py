"""GB300-native grouped / depthwise convolution forward.

The compute path is the CUDA library ``libgconv.so`` (kernels in ``csrc/``,
C ABI in ``include/gconv.h``); this package holds its thin ctypes binding
(``_binding``), the build step (``build``), seeded synthetic workloads
(``inputs``) and the roofline accounting used by the benchmark
(``roofline``).  PyTorch, where used, only provides device memory and
streams.
"""
from ._binding import (  # noqa: F401
    GconvError,
    gconv_device_status,
    gconv_epilogue_apply,
    gconv_last_error,
    gconv_options,
    gconv_problem,
    gconv_status_string,
    grouped_conv_bwd_data,
    grouped_conv_bwd_data_ex,
    grouped_conv_bwd_data_noalloc,
    grouped_conv_bwd_data_route,
    grouped_conv_bwd_weight,
    grouped_conv_bwd_weight_ex,
    grouped_conv_bwd_weight_workspace_size,
    grouped_conv_bwd_data_workspace_size,
    grouped_conv_fwd,
    grouped_conv_fwd_ex,
    grouped_conv_fwd_dw_pw,
    grouped_conv_fwd_dw_pw_ex,
    grouped_conv_fwd_dw_pw_supported,
    grouped_conv_out_shape,
    grouped_conv_select,
    load_library,
    make_problem,
    problem_of,
    DTYPE_CODES,
    KERNEL_NAMES,
)


def conv_forward(x, w, bias, wl, stream=None, out=None):
    """y = grouped_conv(x, w) (+ bias) for device tensors laid out as the
    workload ``wl`` states; allocates y with torch unless ``out`` is given."""
    import torch

    p = problem_of(wl)
    Do, Ho, Wo = grouped_conv_out_shape(p)
    shape = (wl.N, Ho, Wo, wl.G, wl.Kg) if wl.ndim == 2 else (wl.N, Do, Ho, Wo, wl.G, wl.Kg)
    y = out if out is not None else torch.empty(shape, dtype=x.dtype, device=x.device)
    s = stream if stream is not None else torch.cuda.current_stream(x.device)
    grouped_conv_fwd(x, w, bias, y, p, DTYPE_CODES[wl.dtype], s)
    return y
