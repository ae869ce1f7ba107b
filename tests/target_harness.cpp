// Reads "float_bits total" pairs from stdin and prints the coreset target the
// library computes for each (host build of the same header the kernels use).
#include <cstdio>
#include <cstring>

#include "target.h"

int main() {
    unsigned bits;
    long long total;
    while (std::scanf("%u %lld", &bits, &total) == 2) {
        float tp;
        std::memcpy(&tp, &bits, 4);
        std::printf("%lld\n", moestep::coreset_target(tp, total));
    }
    return 0;
}
