/*
 * Run-time compilation of operator source (GPUOS page, §3 Q2 "3. Dynamic
 * Operator Table", step 1: an operator is compiled at run time and injected
 * into the table without restarting the executor).
 *
 * gpuos_compile_op hands CUDA C++ source, prefixed with the operator ABI
 * header below, to NVRTC and returns a relocatable sm_103a cubin: the form
 * gpuos_load_module links into the executor and gpuos_register_op installs.
 * libnvrtc is opened at run time (dlopen), so the library itself does not
 * depend on it. The produced image is only handed on to the driver's linker;
 * nothing here reads or inspects its contents.
 */
#include <dlfcn.h>
#include <nvrtc.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>

#include "gpuos_internal.h"

namespace {

/* The operator ABI, as NVRTC sees it (no system headers there). It must
 * match gpuos_devdesc and gpuos_op_fn of the executor; the sizes are checked
 * by a static_assert compiled into every operator. */
const char kOpHeader[] =
    "typedef unsigned char uint8_t;\n"
    "typedef unsigned short uint16_t;\n"
    "typedef unsigned int uint32_t;\n"
    "typedef int int32_t;\n"
    "typedef unsigned long long uint64_t;\n"
    "struct gpuos_devdesc {\n"
    "    uint16_t op_id; uint8_t dtype; uint8_t flags; uint32_t ntiles;\n"
    "    uint64_t dep[2];\n"
    "    uint64_t a, b, out, aux0, aux1, aux2;\n"
    "    uint32_t dims[6]; float fparam[2];\n"
    "    uint64_t fn; uint64_t ticket; uint32_t version; uint32_t pad;\n"
    "};\n"
    "static_assert(sizeof(gpuos_devdesc) == 128, \"descriptor layout\");\n"
    "typedef int (*gpuos_op_fn)(const gpuos_devdesc *, uint32_t);\n"
    "#define GPUOS_ST_OK 0\n"
    "#define GPUOS_ST_BAD_ARGS 2\n"
    "#define GPUOS_F32 0\n"
    "#define GPUOS_BF16 1\n"
    "/* An operator: __device__ int op(const gpuos_devdesc *d, uint32_t tile),\n"
    " * called by all 32 lanes of one warp with the same arguments, returning a\n"
    " * status identical on every lane; exported through a __device__ variable\n"
    " * of type gpuos_op_fn whose name is given to gpuos_register_op. */\n";

typedef nvrtcResult (*create_t)(nvrtcProgram *, const char *, const char *, int, const char *const *,
                                const char *const *);
typedef nvrtcResult (*destroy_t)(nvrtcProgram *);
typedef nvrtcResult (*compile_t)(nvrtcProgram, int, const char *const *);
typedef nvrtcResult (*size_t_fn)(nvrtcProgram, size_t *);
typedef nvrtcResult (*get_t)(nvrtcProgram, char *);

struct Nvrtc {
    bool ok = false;
    create_t create = nullptr;
    destroy_t destroy = nullptr;
    compile_t compile = nullptr;
    size_t_fn log_size = nullptr, cubin_size = nullptr;
    get_t log = nullptr, cubin = nullptr;
};

const Nvrtc &nvrtc()
{
    static Nvrtc n;
    static std::once_flag once;
    std::call_once(once, [] {
        void *h = nullptr;
        for (const char *name : {"libnvrtc.so.13", "libnvrtc.so"})
            if ((h = dlopen(name, RTLD_NOW | RTLD_LOCAL)) != nullptr) break;
        if (!h) return;
        n.create = reinterpret_cast<create_t>(dlsym(h, "nvrtcCreateProgram"));
        n.destroy = reinterpret_cast<destroy_t>(dlsym(h, "nvrtcDestroyProgram"));
        n.compile = reinterpret_cast<compile_t>(dlsym(h, "nvrtcCompileProgram"));
        n.log_size = reinterpret_cast<size_t_fn>(dlsym(h, "nvrtcGetProgramLogSize"));
        n.log = reinterpret_cast<get_t>(dlsym(h, "nvrtcGetProgramLog"));
        n.cubin_size = reinterpret_cast<size_t_fn>(dlsym(h, "nvrtcGetCUBINSize"));
        n.cubin = reinterpret_cast<get_t>(dlsym(h, "nvrtcGetCUBIN"));
        n.ok = n.create && n.destroy && n.compile && n.log_size && n.log && n.cubin_size && n.cubin;
    });
    return n;
}

void copy_log(nvrtcProgram prog, char *out, size_t cap)
{
    if (!out || cap == 0) return;
    out[0] = 0;
    size_t n = 0;
    if (nvrtc().log_size(prog, &n) != NVRTC_SUCCESS || n == 0) return;
    std::string s(n, '\0');
    if (nvrtc().log(prog, &s[0]) != NVRTC_SUCCESS) return;
    const size_t k = (n < cap) ? n : cap - 1;
    memcpy(out, s.data(), k);
    out[k] = 0;
}

} // namespace

extern "C" {

GPUOS_API const char *gpuos_op_header(void) { return kOpHeader; }

GPUOS_API int gpuos_compile_op(const char *source, const char *name, void **image, size_t *size, char *log,
                               size_t log_cap)
{
    if (log && log_cap) log[0] = 0;
    if (!source || !image || !size) return GPUOS_EINVAL;
    *image = nullptr;
    *size = 0;
    const Nvrtc &n = nvrtc();
    if (!n.ok) {
        if (log && log_cap) snprintf(log, log_cap, "libnvrtc could not be opened");
        return GPUOS_ECUDA;
    }
    const std::string src = std::string(kOpHeader) + source;
    nvrtcProgram prog = nullptr;
    if (n.create(&prog, src.c_str(), name ? name : "gpuos_op.cu", 0, nullptr, nullptr) != NVRTC_SUCCESS)
        return GPUOS_ECUDA;
    /* relocatable (the executor links it), the executor's architecture and
     * per-thread register budget */
    const std::string regs = "--maxrregcount=" + std::to_string(GPUOS_MAX_REGS);
    const char *opts[] = {"--gpu-architecture=sm_103a", "--relocatable-device-code=true", regs.c_str(),
                          "--std=c++17", "-default-device"};
    const nvrtcResult cr = n.compile(prog, (int)(sizeof(opts) / sizeof(opts[0])), opts);
    copy_log(prog, log, log_cap);
    int rc = GPUOS_OK;
    if (cr != NVRTC_SUCCESS) {
        rc = GPUOS_ECOMPILE;
    } else {
        size_t k = 0;
        if (n.cubin_size(prog, &k) != NVRTC_SUCCESS || k == 0) {
            rc = GPUOS_ECUDA;
        } else {
            void *buf = malloc(k);
            if (!buf) {
                rc = GPUOS_ENOMEM;
            } else if (n.cubin(prog, static_cast<char *>(buf)) != NVRTC_SUCCESS) {
                free(buf);
                rc = GPUOS_ECUDA;
            } else {
                *image = buf;
                *size = k;
            }
        }
    }
    n.destroy(&prog);
    return rc;
}

GPUOS_API void gpuos_free_image(void *image) { free(image); }

} // extern "C"
