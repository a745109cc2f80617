// Fused MobileNetV2-style block tail: depthwise 3x3 convolution + bias +
// activation, then a 1x1 projection (C -> K) + bias, in one kernel; the
// depthwise output never leaves the SM.
#pragma once

#include "kernels.h"

namespace gconv {

// Shape limits of the fused kernel: 2D depthwise (G = C, Cg = Kg = 1) with a
// 3x3 filter, dilation 1, equal H / W strides of 1 or 2; C a multiple of 16
// up to 256; K a multiple of 8 up to 256; any H and W; 16-bit data.  act: 0
// none, 1 ReLU, 2 ReLU6.
bool dw_pw_supported(const Geometry& g, DType dt, int K, int act);

// a.x = x, a.w = the depthwise weights, a.bias = the depthwise bias (or
// null), a.y = y [N, Ho, Wo, K]; w_pw [K, C], b_pw [K] (or null).
// a.tile[0..2]: channels per depthwise thread (8 or 4), tile rows, tile
// columns to force (0 = automatic).
// cudaErrorNotSupported when the shape or the pointers' 16-byte alignment
// are outside the kernel, or its shared memory does not fit the device.
cudaError_t dw_pw_launch(const Geometry& g, const LaunchArgs& a, const void* w_pw, const void* b_pw, int K, int act,
                         const DeviceInfo& dev);

}  // namespace gconv
