// decode_launch.cu — the decode kernel instances (format x head_dim x P' terms) and their launchers.
#include "decode.cuh"

namespace kvq {
namespace {

template <int FMT, int D>
DecodeInstance instance_of() {
  using Lo = DecodeLayout<FMT, D>;
  return DecodeInstance{{reinterpret_cast<const void*>(&decode_kernel<FMT, D, true>),
                         reinterpret_cast<const void*>(&decode_kernel<FMT, D, false>)},
                        Lo::kSmemBytes,
                        Lo::kThreads,
                        Lo::kCW,
                        DecodeTraits<FMT, D>::kRow,
                        &decode_head_group<FMT, D>,
                        Lo::kRegSplit ? Lo::kLaunchRegs : 0};
}

template <int FMT, int D>
cudaError_t launch_t(const CUtensorMap& tk, const CUtensorMap& tv, const DecodeParams& p, int grid,
                     cudaStream_t stream) {
  using Lo = DecodeLayout<FMT, D>;
  // programmatic dependent of the preceding kernel: the kernel waits for it
  // (griddepcontrol.wait) before touching anything that kernel may write
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(Lo::kThreads);
  cfg.dynamicSmemBytes = Lo::kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // fp32 output: P' = hi + lo terms; bf16 output: the hi term alone
  return p.out_bf16 ? cudaLaunchKernelEx(&cfg, decode_kernel<FMT, D, false>, tk, tv, p)
                    : cudaLaunchKernelEx(&cfg, decode_kernel<FMT, D, true>, tk, tv, p);
}

}  // namespace

bool decode_instance(int format, int head_dim, DecodeInstance* out) {
  if (format == KVQ_FMT_INT8 && head_dim == 256) *out = instance_of<KVQ_FMT_INT8, 256>();
  else if (format == KVQ_FMT_INT8 && head_dim == 128) *out = instance_of<KVQ_FMT_INT8, 128>();
  else if (format == KVQ_FMT_INT8_G32 && head_dim == 256) *out = instance_of<KVQ_FMT_INT8_G32, 256>();
  else if (format == KVQ_FMT_INT8_G32 && head_dim == 128) *out = instance_of<KVQ_FMT_INT8_G32, 128>();
  else if (format == KVQ_FMT_BF16 && head_dim == 256) *out = instance_of<KVQ_FMT_BF16, 256>();
  else if (format == KVQ_FMT_BF16 && head_dim == 128) *out = instance_of<KVQ_FMT_BF16, 128>();
  else if (format == KVQ_FMT_NVFP4 && head_dim == 256) *out = instance_of<KVQ_FMT_NVFP4, 256>();
  else if (format == KVQ_FMT_NVFP4 && head_dim == 128) *out = instance_of<KVQ_FMT_NVFP4, 128>();
  else return false;
  return true;
}

cudaError_t launch_decode(int format, int head_dim, const CUtensorMap& tk, const CUtensorMap& tv,
                          const DecodeParams& p, int grid, cudaStream_t stream) {
  if (format == KVQ_FMT_INT8 && head_dim == 256) return launch_t<KVQ_FMT_INT8, 256>(tk, tv, p, grid, stream);
  if (format == KVQ_FMT_INT8 && head_dim == 128) return launch_t<KVQ_FMT_INT8, 128>(tk, tv, p, grid, stream);
  if (format == KVQ_FMT_INT8_G32 && head_dim == 256) return launch_t<KVQ_FMT_INT8_G32, 256>(tk, tv, p, grid, stream);
  if (format == KVQ_FMT_INT8_G32 && head_dim == 128) return launch_t<KVQ_FMT_INT8_G32, 128>(tk, tv, p, grid, stream);
  if (format == KVQ_FMT_BF16 && head_dim == 256) return launch_t<KVQ_FMT_BF16, 256>(tk, tv, p, grid, stream);
  if (format == KVQ_FMT_BF16 && head_dim == 128) return launch_t<KVQ_FMT_BF16, 128>(tk, tv, p, grid, stream);
  if (format == KVQ_FMT_NVFP4 && head_dim == 256) return launch_t<KVQ_FMT_NVFP4, 256>(tk, tv, p, grid, stream);
  if (format == KVQ_FMT_NVFP4 && head_dim == 128) return launch_t<KVQ_FMT_NVFP4, 128>(tk, tv, p, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace kvq
